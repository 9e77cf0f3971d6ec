// silu.cu -- the MLP's gated product h = binary16(silu(g) * u) as a kernel of
// its own (the step between the gate/up projections and the down
// projection when it is not fused into the producing kernel), and the
// row interleaving of two packed weight matrices for the fused form.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "silu.cuh"

namespace w4a8 {

namespace {

// h[m * ld_h + i] = silu_mul_h(g[m * ld + i * stride], u[m * ld + i * stride])
// for m < M, i < n.
__global__ void __launch_bounds__(256) silu_mul_kernel(const float* __restrict__ g, const float* __restrict__ u,
                                                       int64_t n, int64_t M, int64_t stride, int64_t ld,
                                                       __half* __restrict__ h) {
    griddep_launch_dependents();
    griddep_wait();  // g and u come from the previous kernel
    const int64_t total = n * M;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = e / n, i = e - m * n;
        const int64_t o = m * ld + i * stride;
        h[e] = silu_mul_h(__ldg(g + o), __ldg(u + o));
    }
}

}  // namespace

cudaError_t launch_silu_mul(const float* g, const float* u, int64_t n, int64_t M, int64_t stride, int64_t ld,
                            uint16_t* h, unsigned flags, cudaStream_t stream) {
    const int64_t total = n * M;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 152 * 8) blocks = 152 * 8;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (flags & 1u) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    __half* hh = reinterpret_cast<__half*>(h);
    return cudaLaunchKernelEx(&cfg, silu_mul_kernel, g, u, n, M, stride, ld, hh);
}

}  // namespace w4a8
