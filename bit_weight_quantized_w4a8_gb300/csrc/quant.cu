// quant.cu -- weight and activation quantizer kernels for sm_103a.
//
// Row-wise and group-wise INT4 weights (the Jetson INT4 page, sections
// 当前实现方式 and 后续优化方向),
// per-channel INT8 weights (the TPU-MLIR W8A16 page, sections 2-3) and the
// dynamic per-row INT8 activation quantizer (the Jetson INT4 page, section
// 正确方向).  One CTA per row: a max|.| reduction over the row, then every
// element is divided by the scale with an IEEE division, rounded half away
// from zero (roundf) and clamped.  These run at load time (weights) or are
// fused into the linear kernel (activations); they are bit-exact, not tuned.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace w4a8 {
namespace {

constexpr int kQThreads = 256;

__device__ __forceinline__ float block_max(float v, float* red) {
    #pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) red[warp] = v;
    __syncthreads();
    float m = 0.f;
    #pragma unroll
    for (int w = 0; w < kQThreads / 32; ++w) m = fmaxf(m, red[w]);
    return m;
}

__device__ __forceinline__ int quant_code(float v, float s, float qmax) {
    if (s == 0.f) return 0;
    float r = roundf(__fdiv_rn(v, s));
    r = fminf(fmaxf(r, -qmax), qmax);
    return static_cast<int>(r);
}

__device__ __forceinline__ float absmax4(float4 v) {
    return fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
}

// W [N][K] fp32 -> Wq [N][K/2] packed nibbles (low nibble = even k), sw [N].
__global__ void __launch_bounds__(kQThreads) w4_quantize_kernel(const float* __restrict__ W,
                                                                 int64_t K,
                                                                 uint8_t* __restrict__ Wq,
                                                                 float* __restrict__ sw) {
    __shared__ float red[kQThreads / 32];
    const int64_t n = blockIdx.x;
    const float4* row = reinterpret_cast<const float4*>(W + n * K);
    float m = 0.f;
    for (int64_t v = threadIdx.x; v < K / 4; v += kQThreads) m = fmaxf(m, absmax4(row[v]));
    const float s = __fdiv_rn(block_max(m, red), 7.f);
    if (threadIdx.x == 0) sw[n] = s;
    uint32_t* out = reinterpret_cast<uint32_t*>(Wq + n * (K / 2));
    for (int64_t u = threadIdx.x; u < K / 8; u += kQThreads) {  // 8 codes -> 4 bytes
        const float4 a = row[2 * u];
        const float4 b = row[2 * u + 1];
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t word = 0;
        #pragma unroll
        for (int t = 0; t < 8; ++t)
            word |= (static_cast<uint32_t>(quant_code(v[t], s, 7.f)) & 0xFu) << (4 * t);
        out[u] = word;
    }
}

// Group-wise INT4 (the Jetson INT4 page, section 后续优化方向: group-wise
// scales): the row-wise rule applied to each group of gs codes of a row.
// W [N][K] fp32 -> Wq [N][K/2] packed nibbles + sg [N][ld] fp32, ld = K/gs
// rounded up to a multiple of 4 (padding written as 0).  One CTA per row,
// one warp per group at a time; gs is a multiple of 32.
__global__ void __launch_bounds__(kQThreads) w4g_quantize_kernel(const float* __restrict__ W,
                                                                  int64_t K, int gs, int64_t ld,
                                                                  uint8_t* __restrict__ Wq,
                                                                  float* __restrict__ sg) {
    const int64_t n = blockIdx.x;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t groups = K / gs;
    for (int64_t g = warp; g < ld; g += kQThreads / 32) {
        if (g >= groups) {
            if (lane == 0) sg[n * ld + g] = 0.f;
            continue;
        }
        const float4* grp = reinterpret_cast<const float4*>(W + n * K + g * gs);
        float m = 0.f;
        for (int v = lane; v < gs / 4; v += 32) m = fmaxf(m, absmax4(grp[v]));
        #pragma unroll
        for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        const float s = __fdiv_rn(m, 7.f);
        if (lane == 0) sg[n * ld + g] = s;
        uint32_t* out = reinterpret_cast<uint32_t*>(Wq + n * (K / 2) + g * (gs / 2));
        for (int u = lane; u < gs / 8; u += 32) {  // 8 codes -> 4 bytes
            const float4 a = grp[2 * u];
            const float4 b = grp[2 * u + 1];
            const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            uint32_t word = 0;
            #pragma unroll
            for (int t = 0; t < 8; ++t)
                word |= (static_cast<uint32_t>(quant_code(v[t], s, 7.f)) & 0xFu) << (4 * t);
            out[u] = word;
        }
    }
}

// W [N][K] fp32 -> Wq8 [N][K] int8 codes taken with the binary16 scale.
__global__ void __launch_bounds__(kQThreads) w8_quantize_kernel(const float* __restrict__ W,
                                                                 int64_t K,
                                                                 int8_t* __restrict__ Wq8,
                                                                 __half* __restrict__ sw16) {
    __shared__ float red[kQThreads / 32];
    const int64_t n = blockIdx.x;
    const float4* row = reinterpret_cast<const float4*>(W + n * K);
    float m = 0.f;
    for (int64_t v = threadIdx.x; v < K / 4; v += kQThreads) m = fmaxf(m, absmax4(row[v]));
    const __half h = __float2half_rn(__fdiv_rn(block_max(m, red), 127.f));
    const float s = __half2float(h);
    if (threadIdx.x == 0) sw16[n] = h;
    uint2* out = reinterpret_cast<uint2*>(Wq8 + n * K);
    for (int64_t u = threadIdx.x; u < K / 8; u += kQThreads) {
        const float4 a = row[2 * u];
        const float4 b = row[2 * u + 1];
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t w[2] = {0u, 0u};
        #pragma unroll
        for (int t = 0; t < 8; ++t)
            w[t >> 2] |= (static_cast<uint32_t>(quant_code(v[t], s, 127.f)) & 0xFFu) << (8 * (t & 3));
        out[u] = make_uint2(w[0], w[1]);
    }
}

// X [M][K] binary16 -> Xq [M][K] int8 + sa [M].
__global__ void __launch_bounds__(kQThreads) act_quantize_kernel(const __half* __restrict__ X,
                                                                  int64_t K,
                                                                  int8_t* __restrict__ Xq,
                                                                  float* __restrict__ sa) {
    __shared__ float red[kQThreads / 32];
    const int64_t m = blockIdx.x;
    const uint4* row = reinterpret_cast<const uint4*>(X + m * K);
    float mx = 0.f;
    for (int64_t v = threadIdx.x; v < K / 8; v += kQThreads) {
        const uint4 h = row[v];
        const __half2* p = reinterpret_cast<const __half2*>(&h);
        #pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float2 f = __half22float2(p[t]);
            mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
    }
    const float s = __fdiv_rn(block_max(mx, red), 127.f);
    if (threadIdx.x == 0) sa[m] = s;
    uint2* out = reinterpret_cast<uint2*>(Xq + m * K);
    for (int64_t v = threadIdx.x; v < K / 8; v += kQThreads) {
        const uint4 h = row[v];
        const __half2* p = reinterpret_cast<const __half2*>(&h);
        uint32_t w[2] = {0u, 0u};
        #pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float2 f = __half22float2(p[t]);
            w[t >> 1] |= (static_cast<uint32_t>(quant_code(f.x, s, 127.f)) & 0xFFu) << (16 * (t & 1));
            w[t >> 1] |= (static_cast<uint32_t>(quant_code(f.y, s, 127.f)) & 0xFFu) << (16 * (t & 1) + 8);
        }
        out[v] = make_uint2(w[0], w[1]);
    }
}

}  // namespace

cudaError_t launch_w4_quantize(const float* W, int64_t N, int64_t K, uint8_t* Wq, float* sw,
                               cudaStream_t stream) {
    w4_quantize_kernel<<<dim3((unsigned)N), kQThreads, 0, stream>>>(W, K, Wq, sw);
    return cudaGetLastError();
}

cudaError_t launch_w4g_quantize(const float* W, int64_t N, int64_t K, int gs, int64_t ld,
                                uint8_t* Wq, float* sg, cudaStream_t stream) {
    w4g_quantize_kernel<<<dim3((unsigned)N), kQThreads, 0, stream>>>(W, K, gs, ld, Wq, sg);
    return cudaGetLastError();
}

cudaError_t launch_w8_quantize(const float* W, int64_t N, int64_t K, int8_t* Wq8, uint16_t* sw16,
                               cudaStream_t stream) {
    w8_quantize_kernel<<<dim3((unsigned)N), kQThreads, 0, stream>>>(
        W, K, Wq8, reinterpret_cast<__half*>(sw16));
    return cudaGetLastError();
}

cudaError_t launch_act_quantize(const uint16_t* X, int64_t M, int64_t K, int8_t* Xq, float* sa,
                                cudaStream_t stream) {
    act_quantize_kernel<<<dim3((unsigned)M), kQThreads, 0, stream>>>(
        reinterpret_cast<const __half*>(X), K, Xq, sa);
    return cudaGetLastError();
}

}  // namespace w4a8
