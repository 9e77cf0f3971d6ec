// isx.cu -- IndexSoftmax for sm_103a (the IntAttention page, section
// 基准/方法设计: IndexSoftmax's three mechanisms).
//
// Per row of int32 logits: delta = rowMax - a, clipped at c_int; a 2^b-entry
// UINT8 exponent table indexed by idx = round(delta' * (2^b - 1) / c_int);
// P = round(255 * E / rowSum(E)) as UINT8.  All of it is integer arithmetic,
// bit-identical to the CPU definition.
//
// HBM-bound (4 bytes in, 1 byte out per element), one pass over HBM: one
// CTA per row keeps the row in registers (up to 8192 elements), takes the
// block max, the per-element table index (kept in registers as bytes), the
// block sum, then writes P from a per-row table of the 2^b possible
// probabilities, round(255 * LUT[i] / S), built once per row.  Rows longer
// than that stream through global memory three times instead.
//
// The index is exact without a division per element: idx is the number of
// k in 1..top with delta' >= T[k], T[k] = ceil(c_int (2k - 1) / (2 top)) (the
// smallest delta' that rounds to k or more).  The fp32 quotient
// x = delta' * top / c_int is within 5e-5 of the exact one, so the exact
// index round(x) is floor(x) or floor(x) + 1 (or exactly floor(x) + 1 past a
// half near an integer), and the single threshold T[floor(x) + 1] decides.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>

#include "kernels.h"

namespace w4a8 {
namespace {

constexpr int kIsxThreads = 256;
constexpr int kIsxWarps = kIsxThreads / 32;

struct IsxArgs {
    const int32_t* A;
    uint8_t* P;
    int64_t rows;
    int cols;
    uint32_t c_int;
    int top;                   // 2^b - 1
    float inv;                 // top / c_int (0 when c_int == 0)
    uint32_t thr[kIsxMaxEntries + 1];  // T[0] = 0, T[1..top], T[top + 1] = UINT32_MAX
    uint8_t lut[kIsxMaxEntries];
};

__device__ __forceinline__ int warp_max_i(int v) {
    #pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

__device__ __forceinline__ int warp_sum_i(int v) {
    #pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Block-wide max / sum over kIsxThreads threads (every thread gets the result).
__device__ __forceinline__ int block_max_i(int v, int* red) {
    v = warp_max_i(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    int m = red[0];
    #pragma unroll
    for (int w = 1; w < kIsxWarps; ++w) m = max(m, red[w]);
    __syncthreads();  // red is reused
    return m;
}

__device__ __forceinline__ int block_sum_i(int v, int* red) {
    v = warp_sum_i(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    int s = 0;
    #pragma unroll
    for (int w = 0; w < kIsxWarps; ++w) s += red[w];
    __syncthreads();
    return s;
}

// The exact table index of one logit given the row max.
__device__ __forceinline__ uint32_t isx_index(int a, int mx, uint32_t c_int, float inv, int top,
                                              const uint32_t* thr) {
    const uint32_t delta = (uint32_t)mx - (uint32_t)a;  // mx >= a: exact as uint32
    const uint32_t cl = delta < c_int ? delta : c_int;
    // x = cl * top / c_int within 5e-5: the exact index is floor(x) or
    // floor(x) + 1, decided by the one threshold between them
    const float x = __uint2float_rn(cl) * inv;
    const int j = min((int)x + 1, top);  // x >= 0: truncation is floor
    return cl >= thr[j] ? (uint32_t)j : (uint32_t)(j - 1);
}

// Stages the launch's table, thresholds into shared memory.
__device__ __forceinline__ void isx_stage(const IsxArgs& a, uint32_t* thr_s, int* lut_s) {
    for (int i = threadIdx.x; i <= a.top + 1; i += kIsxThreads) thr_s[i] = a.thr[i];
    for (int i = threadIdx.x; i <= a.top; i += kIsxThreads) lut_s[i] = a.lut[i];
}

// Register-resident rows: each thread holds Q accesses of V consecutive
// logits (V = 4: one 16-byte load, one 4-byte store of P; V = 1 otherwise).
template <int V, int Q>
__global__ void __launch_bounds__(kIsxThreads) isx_rows_kernel(const __grid_constant__ IsxArgs a) {
    __shared__ uint32_t thr_s[kIsxMaxEntries + 1];
    __shared__ int lut_s[kIsxMaxEntries];
    __shared__ int ptab_s[kIsxMaxEntries];
    __shared__ int red[kIsxWarps];
    isx_stage(a, thr_s, lut_s);
    __syncthreads();

    const int nacc = a.cols / V;  // accesses per row (cols % V == 0)
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        const int32_t* Ar = a.A + r * a.cols;
        int x[Q][V];
        int mx = INT32_MIN;
        #pragma unroll
        for (int q = 0; q < Q; ++q) {
            const int k = threadIdx.x + q * kIsxThreads;
            if (k < nacc) {
                if constexpr (V == 4) {
                    const int4 v = __ldcs(reinterpret_cast<const int4*>(Ar) + k);
                    x[q][0] = v.x; x[q][1] = v.y; x[q][2] = v.z; x[q][3] = v.w;
                } else {
                    x[q][0] = __ldcs(Ar + k);
                }
                #pragma unroll
                for (int u = 0; u < V; ++u) mx = max(mx, x[q][u]);
            }
        }
        mx = block_max_i(mx, red);

        uint32_t idx[Q];  // V table indices per access, one byte each
        int sum = 0;
        #pragma unroll
        for (int q = 0; q < Q; ++q) {
            idx[q] = 0;
            const int k = threadIdx.x + q * kIsxThreads;
            if (k < nacc) {
                #pragma unroll
                for (int u = 0; u < V; ++u) {
                    const uint32_t i = isx_index(x[q][u], mx, a.c_int, a.inv, a.top, thr_s);
                    sum += lut_s[i];
                    idx[q] |= i << (8 * u);
                }
            }
        }
        const int S = block_sum_i(sum, red);  // >= LUT[0] > 0 (the max's entry)
        // the 2^b possible probabilities of this row, round(255 E / S) with
        // halves up, in uint32 (2 S < 2^32 for every row the ABI admits)
        for (int i = threadIdx.x; i <= a.top; i += kIsxThreads)
            ptab_s[i] = (int)((2u * 255u * (uint32_t)lut_s[i] + (uint32_t)S) / (2u * (uint32_t)S));
        __syncthreads();

        uint8_t* Pr = a.P + r * a.cols;
        #pragma unroll
        for (int q = 0; q < Q; ++q) {
            const int k = threadIdx.x + q * kIsxThreads;
            if (k < nacc) {
                if constexpr (V == 4) {
                    const uint32_t w = (uint32_t)ptab_s[idx[q] & 0xFF] |
                                       ((uint32_t)ptab_s[(idx[q] >> 8) & 0xFF] << 8) |
                                       ((uint32_t)ptab_s[(idx[q] >> 16) & 0xFF] << 16) |
                                       ((uint32_t)ptab_s[idx[q] >> 24] << 24);
                    __stcs(reinterpret_cast<uint32_t*>(Pr) + k, w);
                } else {
                    Pr[k] = (uint8_t)ptab_s[idx[q] & 0xFF];
                }
            }
        }
        __syncthreads();  // ptab_s is rebuilt for the next row
    }
}

// Rows too long for registers: max, then sum, then output, each streaming
// the row from global memory.
__global__ void __launch_bounds__(kIsxThreads) isx_long_kernel(const __grid_constant__ IsxArgs a) {
    __shared__ uint32_t thr_s[kIsxMaxEntries + 1];
    __shared__ int lut_s[kIsxMaxEntries];
    __shared__ int ptab_s[kIsxMaxEntries];
    __shared__ int red[kIsxWarps];
    isx_stage(a, thr_s, lut_s);
    __syncthreads();
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        const int32_t* Ar = a.A + r * a.cols;
        int mx = INT32_MIN;
        for (int k = threadIdx.x; k < a.cols; k += kIsxThreads) mx = max(mx, Ar[k]);
        mx = block_max_i(mx, red);
        int sum = 0;
        for (int k = threadIdx.x; k < a.cols; k += kIsxThreads)
            sum += lut_s[isx_index(Ar[k], mx, a.c_int, a.inv, a.top, thr_s)];
        const int S = block_sum_i(sum, red);
        for (int i = threadIdx.x; i <= a.top; i += kIsxThreads)
            ptab_s[i] = (int)((2u * 255u * (uint32_t)lut_s[i] + (uint32_t)S) / (2u * (uint32_t)S));
        __syncthreads();
        uint8_t* Pr = a.P + r * a.cols;
        for (int k = threadIdx.x; k < a.cols; k += kIsxThreads)
            Pr[k] = (uint8_t)ptab_s[isx_index(Ar[k], mx, a.c_int, a.inv, a.top, thr_s)];
        __syncthreads();
    }
}

template <int V>
cudaError_t launch_rows(const IsxArgs& a, int q_needed, dim3 grid, cudaStream_t stream) {
    if (q_needed <= 1) isx_rows_kernel<V, 1><<<grid, kIsxThreads, 0, stream>>>(a);
    else if (q_needed <= 2) isx_rows_kernel<V, 2><<<grid, kIsxThreads, 0, stream>>>(a);
    else if (q_needed <= 4) isx_rows_kernel<V, 4><<<grid, kIsxThreads, 0, stream>>>(a);
    else isx_rows_kernel<V, 8><<<grid, kIsxThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

void isx_build_lut(int b, double c, uint8_t* lut) {
    const int n = 1 << b;
    for (int i = 0; i < n - 1; ++i)
        lut[i] = (uint8_t)std::round(255.0 * std::exp(-c * (double)i / (double)(n - 1)));
    lut[n - 1] = 0;
}

int64_t isx_c_int(double c, int64_t d, float s_q, float s_k) {
    return (int64_t)std::llround(c * std::sqrt((double)d) / ((double)s_q * (double)s_k));
}

void isx_thresholds(uint32_t c_int, int b, uint32_t* thr) {
    const int top = (1 << b) - 1;
    thr[0] = 0;
    for (int k = 1; k <= top; ++k) {
        // smallest delta' with (2 delta' top + c) / (2 c) >= k, i.e. ceil(c (2k - 1) / (2 top));
        // with c = 0 no distance reaches index 1
        const uint64_t num = (uint64_t)c_int * (uint64_t)(2 * k - 1);
        thr[k] = c_int == 0 ? UINT32_MAX : (uint32_t)((num + 2 * top - 1) / (2 * top));
    }
    thr[top + 1] = UINT32_MAX;
}

int isx_kernel_kind(int64_t cols, bool vec_ok, int* q_needed) {
    const int V = vec_ok ? 4 : 1;
    const int64_t acc = cols / V;
    const int64_t q = (acc + kIsxThreads - 1) / kIsxThreads;
    *q_needed = (int)q;
    if (q <= 8) return vec_ok ? 4 : 1;
    return 0;  // streaming kernel
}

cudaError_t launch_index_softmax(const int32_t* A, int64_t rows, int64_t cols, uint32_t c_int,
                                 int b, const uint8_t* lut, const uint32_t* thr, uint8_t* P,
                                 cudaStream_t stream) {
    IsxArgs a = {};
    a.A = A;
    a.P = P;
    a.rows = rows;
    a.cols = (int)cols;
    a.c_int = c_int;
    a.top = (1 << b) - 1;
    a.inv = c_int > 0 ? (float)a.top / (float)c_int : 0.f;
    for (int i = 0; i <= a.top + 1; ++i) a.thr[i] = thr[i];
    for (int i = 0; i <= a.top; ++i) a.lut[i] = lut[i];
    const bool vec_ok = (cols % 4 == 0) && (reinterpret_cast<uintptr_t>(A) % 16 == 0) &&
                        (reinterpret_cast<uintptr_t>(P) % 4 == 0);
    int q = 0;
    const int kind = isx_kernel_kind(cols, vec_ok, &q);
    const dim3 grid((unsigned)(rows < 0x7FFFFFFF ? rows : 0x7FFFFFFF));
    if (kind == 4) return launch_rows<4>(a, q, grid, stream);
    if (kind == 1) return launch_rows<1>(a, q, grid, stream);
    isx_long_kernel<<<grid, kIsxThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace w4a8
