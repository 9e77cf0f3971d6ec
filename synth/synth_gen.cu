// synth_gen.cu -- the seeded input generator of synth/__init__.py as a CUDA
// kernel, for weight tensors too large to draw on the host.  Same counter
// arithmetic, same Irwin-Hall(12) sum, one fp32 multiply: identical bits.
// Test and benchmark infrastructure; not part of the library.
#include <cuda_runtime.h>

#include <cstdint>

namespace {

__device__ __forceinline__ uint32_t fmix32(uint32_t h) {
    h ^= h >> 16;
    h *= 0x85EBCA6Bu;
    h ^= h >> 13;
    h *= 0xC2B2AE35u;
    h ^= h >> 16;
    return h;
}

__global__ void normal_kernel(uint32_t key, uint64_t offset, uint64_t count, float sigma,
                              float* __restrict__ out) {
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t e = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; e < count; e += stride) {
        const uint32_t i = (uint32_t)(offset + e);
        const uint32_t a = fmix32(i ^ key);
        int32_t s = 0;
        #pragma unroll
        for (uint32_t j = 0; j < 6; ++j) {
            const uint32_t w = fmix32(a + (j + 1u) * 0x9E3779B9u);
            s += (int32_t)(w & 0xFFFFu) + (int32_t)(w >> 16);
        }
        const float z = __fmul_rn((float)(s - 393210), 1.0f / 65536.0f);
        out[e] = __fmul_rn(z, sigma);
    }
}

uint32_t fmix32_host(uint32_t h) {
    h ^= h >> 16;
    h *= 0x85EBCA6Bu;
    h ^= h >> 13;
    h *= 0xC2B2AE35u;
    h ^= h >> 16;
    return h;
}

}  // namespace

extern "C" int synth_normal_f32(uint32_t seed, uint64_t offset, uint64_t count, float sigma,
                                float* out, void* stream) {
    if (count == 0) return 0;
    if (offset + count > (1ull << 32)) return 3;  // counters are 32-bit
    int blocks = (int)((count + 255) / 256);
    if (blocks > 152 * 32) blocks = 152 * 32;
    normal_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(fmix32_host(seed), offset, count, sigma, out);
    return cudaGetLastError() == cudaSuccess ? 0 : 5;
}
