// silu.cuh -- the gated product of the MLP between the gate/up projections
// and the down projection, h = binary16(silu(g) * u), shared by the fused
// epilogue of the one-row GEMV and the stand-alone kernel.
#pragma once

#include <cuda_fp16.h>

namespace w4a8 {

// silu(g) * u = g / (1 + exp(-g)) * u in fp32: expf (CUDA's accurate single
// precision exp, within 2 ulp), then one IEEE add, one IEEE division, one
// IEEE multiply, and one round-to-nearest-even conversion to binary16.  The
// fp32 value is within 2^-20 |v| of v = silu(g) * u in exact arithmetic, so
// its binary16 rounding is that of v unless v lies that close to a binary16
// rounding boundary.
__device__ __forceinline__ __half silu_mul_h(float g, float u) {
    const float e = expf(-g);
    return __float2half_rn(__fmul_rn(__fdiv_rn(g, __fadd_rn(1.f, e)), u));
}

}  // namespace w4a8
