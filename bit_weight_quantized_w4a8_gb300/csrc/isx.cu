// isx.cu -- IndexSoftmax for sm_103a (the IntAttention page, section
// 基准/方法设计: IndexSoftmax's three mechanisms).
//
// Per row of int32 logits: delta = rowMax - a, clipped at c_int; a 2^b-entry
// UINT8 exponent table indexed by idx = round(delta' * (2^b - 1) / c_int);
// P = round(255 * E / rowSum(E)) as UINT8.  All of it is integer arithmetic,
// bit-identical to the CPU definition.
//
// HBM-bound (4 bytes in, 1 byte out per element), one pass over HBM: one
// CTA of 128 threads per row keeps the row in registers (up to 8192
// elements; 128 threads leave each thread enough elements to amortize the
// per-row reductions, 256 or 64 were measured slower), takes the
// block max, the per-element table index (kept in registers as bytes), the
// block sum, then writes P from a per-row table of the 2^b possible
// probabilities, round(255 * LUT[i] / S), built once per row.  Rows longer
// than that stream through global memory three times instead.
//
// The index is exact without a division per element: idx is the number of
// k in 1..top with delta' >= T[k], T[k] = ceil(c_int (2k - 1) / (2 top)) (the
// smallest delta' that rounds to k or more).  An integer estimate
// e = floor(delta' M / 2^32), M = ceil(2^32 top / c_int), is never below
// floor(x), x = delta' top / c_int, and less than 1/2 above it, so the index
// round(x) is e or e + 1 and the single threshold T[e + 1] decides; it is
// packed with LUT[e] and LUT[e + 1] into one 8-byte shared-memory entry.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>

#include "kernels.h"

namespace w4a8 {
namespace {

constexpr int kIsxThreads = 128;
constexpr int kIsxWarps = kIsxThreads / 32;

struct IsxArgs {
    const int32_t* A;
    uint8_t* P;
    int64_t rows;
    int cols;
    uint32_t c_int;
    int top;                   // 2^b - 1
    uint32_t m_hi, m_lo;       // M = ceil(2^32 top / c_int) = m_hi 2^32 + m_lo (0 when c_int == 0)
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

// Shared table entry e (0 <= e <= top): T[e + 1], and LUT[e] | LUT[e + 1] << 8.
__device__ __forceinline__ void isx_stage(const IsxArgs& a, uint2* tab) {
    for (int e = threadIdx.x; e <= a.top; e += kIsxThreads) {
        const uint32_t next = e < a.top ? a.lut[e + 1] : 0u;
        tab[e] = make_uint2(a.thr[e + 1], (uint32_t)a.lut[e] | (next << 8));
    }
}

// The exact table index of one logit given the row max, and its entry E.
// e = floor(cl M / 2^32) never undershoots floor(x), x = cl top / c_int, and
// exceeds it by less than 1/2, so the index round(x) is e or e + 1 and
// T[e + 1] decides (when e = floor(x) + 1, x is past its half and T[e + 1]
// is out of reach).
// kHi = false: M < 2^32 (m_hi = 0, every c_int >= top), one multiply-high.
template <bool kHi = true>
__device__ __forceinline__ uint32_t isx_lookup(int a, int mx, uint32_t c_int, uint32_t m_hi,
                                               uint32_t m_lo, const uint2* tab, int* E) {
    const uint32_t delta = (uint32_t)mx - (uint32_t)a;  // mx >= a: exact as uint32
    const uint32_t cl = delta < c_int ? delta : c_int;
    const uint32_t e = (kHi ? cl * m_hi : 0u) + __umulhi(cl, m_lo);  // <= top: no overflow
    const uint2 t = tab[e];
    const bool up = cl >= t.x;
    *E = (int)__byte_perm(t.y, 0u, up ? 0x4441u : 0x4440u);
    return up ? e + 1u : e;
}

// Register-resident rows: each thread holds Q accesses of V consecutive
// logits (V = 4: one 16-byte load, one 4-byte store of P; V = 1 otherwise).
// Three barriers per row: the reduction slots and the probability table are
// double-buffered by row parity, so no row waits for the previous one's
// readers (a thread two rows ahead has passed barriers every other thread
// reached only after finishing those reads).
template <int V, int Q, bool kHi>
__global__ void __launch_bounds__(kIsxThreads) isx_rows_kernel(const __grid_constant__ IsxArgs a) {
    __shared__ uint2 tab_s[kIsxMaxEntries];
    __shared__ int ptab_s[2][kIsxMaxEntries];
    __shared__ int red_max[2][kIsxWarps];
    __shared__ int red_sum[2][kIsxWarps];
    isx_stage(a, tab_s);
    __syncthreads();

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nacc = a.cols / V;  // accesses per row (cols % V == 0)
    int par = 0;
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x, par ^= 1) {
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
        mx = warp_max_i(mx);
        if (lane == 0) red_max[par][warp] = mx;
        __syncthreads();
        mx = red_max[par][0];
        #pragma unroll
        for (int w = 1; w < kIsxWarps; ++w) mx = max(mx, red_max[par][w]);

        uint32_t idx[Q];  // V table indices per access, one byte each
        int sum = 0;
        #pragma unroll
        for (int q = 0; q < Q; ++q) {
            idx[q] = 0;
            const int k = threadIdx.x + q * kIsxThreads;
            if (k < nacc) {
                #pragma unroll
                for (int u = 0; u < V; ++u) {
                    int E;
                    const uint32_t i = isx_lookup<kHi>(x[q][u], mx, a.c_int, a.m_hi, a.m_lo, tab_s, &E);
                    sum += E;
                    idx[q] |= i << (8 * u);
                }
            }
        }
        sum = warp_sum_i(sum);
        if (lane == 0) red_sum[par][warp] = sum;
        __syncthreads();
        int S = 0;  // >= LUT[0] > 0 (the max's entry)
        #pragma unroll
        for (int w = 0; w < kIsxWarps; ++w) S += red_sum[par][w];
        // the 2^b possible probabilities of this row, round(255 E / S) with
        // halves up, in uint32 (2 S < 2^32 for every row the ABI admits)
        for (int i = threadIdx.x; i <= a.top; i += kIsxThreads)
            ptab_s[par][i] = (int)((2u * 255u * (tab_s[i].y & 0xFFu) + (uint32_t)S) / (2u * (uint32_t)S));
        __syncthreads();

        const int* pt = ptab_s[par];
        uint8_t* Pr = a.P + r * a.cols;
        #pragma unroll
        for (int q = 0; q < Q; ++q) {
            const int k = threadIdx.x + q * kIsxThreads;
            if (k < nacc) {
                if constexpr (V == 4) {
                    const uint32_t w = (uint32_t)pt[idx[q] & 0xFF] |
                                       ((uint32_t)pt[(idx[q] >> 8) & 0xFF] << 8) |
                                       ((uint32_t)pt[(idx[q] >> 16) & 0xFF] << 16) |
                                       ((uint32_t)pt[idx[q] >> 24] << 24);
                    __stcs(reinterpret_cast<uint32_t*>(Pr) + k, w);
                } else {
                    Pr[k] = (uint8_t)pt[idx[q] & 0xFF];
                }
            }
        }
    }
}

// Rows too long for registers: max, then sum, then output, each streaming
// the row from global memory (same barrier scheme).
__global__ void __launch_bounds__(kIsxThreads) isx_long_kernel(const __grid_constant__ IsxArgs a) {
    __shared__ uint2 tab_s[kIsxMaxEntries];
    __shared__ int ptab_s[2][kIsxMaxEntries];
    __shared__ int red_max[2][kIsxWarps];
    __shared__ int red_sum[2][kIsxWarps];
    isx_stage(a, tab_s);
    __syncthreads();
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int par = 0;
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x, par ^= 1) {
        const int32_t* Ar = a.A + r * a.cols;
        int mx = INT32_MIN;
        for (int k = threadIdx.x; k < a.cols; k += kIsxThreads) mx = max(mx, Ar[k]);
        mx = warp_max_i(mx);
        if (lane == 0) red_max[par][warp] = mx;
        __syncthreads();
        mx = red_max[par][0];
        for (int w = 1; w < kIsxWarps; ++w) mx = max(mx, red_max[par][w]);
        int sum = 0;
        for (int k = threadIdx.x; k < a.cols; k += kIsxThreads) {
            int E;
            isx_lookup(Ar[k], mx, a.c_int, a.m_hi, a.m_lo, tab_s, &E);
            sum += E;
        }
        sum = warp_sum_i(sum);
        if (lane == 0) red_sum[par][warp] = sum;
        __syncthreads();
        int S = 0;
        for (int w = 0; w < kIsxWarps; ++w) S += red_sum[par][w];
        for (int i = threadIdx.x; i <= a.top; i += kIsxThreads)
            ptab_s[par][i] = (int)((2u * 255u * (tab_s[i].y & 0xFFu) + (uint32_t)S) / (2u * (uint32_t)S));
        __syncthreads();
        uint8_t* Pr = a.P + r * a.cols;
        for (int k = threadIdx.x; k < a.cols; k += kIsxThreads) {
            int E;
            Pr[k] = (uint8_t)ptab_s[par][isx_lookup(Ar[k], mx, a.c_int, a.m_hi, a.m_lo, tab_s, &E)];
        }
    }
}

template <int V, bool kHi>
cudaError_t launch_rows_hi(const IsxArgs& a, int q_needed, dim3 grid, cudaStream_t stream) {
    if (q_needed <= 1) isx_rows_kernel<V, 1, kHi><<<grid, kIsxThreads, 0, stream>>>(a);
    else if (q_needed <= 2) isx_rows_kernel<V, 2, kHi><<<grid, kIsxThreads, 0, stream>>>(a);
    else if (q_needed <= 4) isx_rows_kernel<V, 4, kHi><<<grid, kIsxThreads, 0, stream>>>(a);
    else if (q_needed <= 8) isx_rows_kernel<V, 8, kHi><<<grid, kIsxThreads, 0, stream>>>(a);
    else isx_rows_kernel<V, 16, kHi><<<grid, kIsxThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

template <int V>
cudaError_t launch_rows(const IsxArgs& a, int q_needed, dim3 grid, cudaStream_t stream) {
    return a.m_hi ? launch_rows_hi<V, true>(a, q_needed, grid, stream)
                  : launch_rows_hi<V, false>(a, q_needed, grid, stream);
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
    if (q <= (vec_ok ? 16 : 8)) return vec_ok ? 4 : 1;
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
    // M = ceil(2^32 top / c_int) < 2^40
    const uint64_t m = c_int > 0 ? (((uint64_t)a.top << 32) + c_int - 1) / c_int : 0;
    a.m_hi = (uint32_t)(m >> 32);
    a.m_lo = (uint32_t)m;
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
