// mma.cu -- W4A8 linear on the sm_103a tensor cores, for decode batches
// where the dp4a GEMV turns ALU-bound (the skinny-batch regime, 2..64 rows).
//
// The arithmetic is the W4A8 contract of the Jetson INT4 page (sections
// 正确方向 / 当前实现方式): INT8 activation codes times INT4 weight codes,
// summed exactly in integers, y = ((float)acc * s_w) * s_a.  Both code sets
// are small integers and so exact in binary16; tcgen05.mma kind::f16 multiplies
// them exactly and accumulates in fp32 in TMEM.  Every partial sum of one
// K piece is an integer of magnitude <= 8 * 127 * 16384 < 2^24, so the fp32
// accumulator holds it exactly whatever the summation order; pieces are
// summed as int32 in a fixed order.  The result is bit-identical to the
// integer definition.
//
// Two kernels:
//  * act_codes_kernel (one CTA per activation row): the per-row INT8
//    quantization (max|x|, s_a = max/127, IEEE division, round half away,
//    clamp), written as binary16 codes for the tensor cores (plus the
//    optional int8 codes and scale outputs); or, for the unfused entry,
//    the given int8 codes widened to binary16.
//  * mma_kernel: one CTA per 128 weight rows and K piece.  Warp 0 streams
//    packed INT4 tiles (128 rows x 64 K = 4 KB) with 2-D TMA into a deep
//    ring; warp 2 streams the binary16 activation tiles (TMA, 128-byte
//    swizzle) into their own ring; warp 1 issues the MMAs (M = 128 weight
//    rows, N = 16..64 batch rows, K = 16, four per tile) into a TMEM
//    accumulator; warps 3-10 widen each weight row's INT4 codes to binary16
//    (two nibbles at a time masked into the mantissa of 1024.0, in a K
//    order permuted inside each 8-code group, as are the activations) straight into
//    TMEM, where the MMA reads its A operand (so the widened weights never
//    pass through shared memory, whose bandwidth would otherwise bound the
//    kernel), then read the accumulator back (tcgen05.ld), convert to
//    int32 and rescale, or store int32 partials for the split-K sum.  Every
//    ring slot is handed back by a tcgen05.commit, so no thread waits for
//    one MMA to finish before issuing the next.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "actq.cuh"
#include "kernels.h"
#include "plan.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace w4a8 {

__device__ unsigned g_mma_error;  // wait timeouts of the tensor-core path (same bits)

namespace {

constexpr int kTileRows = 128;                  // weight rows per CTA (MMA M)
constexpr int kKBlock = 64;                     // K block: 128 bytes of bf16 per row
constexpr int kStageK = 2;                      // K blocks per pipeline stage (8 MMAs, one commit)
constexpr int kWBlocks = 4;                     // K blocks per weight load: 128 bytes of a row
constexpr int kWStages = 3;                     // packed INT4 ring (16 KB a load)
constexpr int kStages = 3;                      // stage ring: A in TMEM, B in shared memory
constexpr int kConvGroups = 2;                  // converter warp groups, alternating stages
constexpr int kConvWarps = 4 * kConvGroups;     // one warp per TMEM lane quarter per group
constexpr int kFirstConvWarp = 3;
constexpr int kMmaThreads = (kFirstConvWarp + kConvWarps) * 32;
constexpr int kWTileBytes = kTileRows * kKBlock / 2 * kWBlocks;  // 16384
constexpr int kBTileMax = 64 * kKBlock * 2;     // one K block of 64 batch rows: 8192
constexpr int kBStageMax = kStageK * kBTileMax;
constexpr uint32_t kTmemCols = 256;             // D: columns 0..63; A stage s: 64 + 64 s
constexpr uint32_t kTmemA = 64;
constexpr uint32_t kTmemAStage = 32 * kStageK;  // two bf16 per column
constexpr int kOffB = 0;
constexpr int kOffW = kOffB + kStages * kBStageMax;
constexpr int kOffBars = kOffW + kWStages * kWTileBytes;
constexpr int kNumBars = 2 * kWStages + 3 * kStages + 5;  // + accfull, dfull[2], dfree[2]
constexpr int kOffMisc = kOffBars + kNumBars * 8;
constexpr int kOffSaSum = kOffMisc + 16;       // e4m3 path: exact code sums of the batch rows
constexpr int kMmaSmem = kOffSaSum + 256 + 1024;  // + slack to align the base to 1024
constexpr int kAQThreads = 256;
// Group scales: the most workspace the chunk sums of a split call may take.
constexpr size_t kGroupPartBytes = 32u << 20;
// Row-wise split K: up to this many pieces store int32 slices that the last
// CTA of a tile adds to the sums it holds; more pieces add into one int32
// accumulator per tile with atomics (the reduction spread over every CTA),
// which the last CTA reads and clears.
constexpr int kSliceMaxP = 3;

static_assert(kWBlocks % kStageK == 0, "stage geometry");
static_assert(kOffB % 1024 == 0 && kOffW % 1024 == 0, "swizzled tiles need 1024-byte alignment");
static_assert(kTmemA + kTmemAStage * kStages <= kTmemCols, "TMEM budget");
// Group scales: D (the integer sums of one group) at columns 0..63 -- two
// buffers of 32 columns when the batch has at most 32 rows --, F (the fp32
// running sums) at 64..127, two A stages at 128 + 64 s.
constexpr int kStagesG = 2;
constexpr uint32_t kTmemF = 64;
constexpr uint32_t kTmemAG = 128;
static_assert(kTmemAG + kTmemAStage * kStagesG <= kTmemCols, "TMEM budget (group scales)");
// e4m3 path: D (2 x 64 columns: W.A_hi, W.A_lo) at 0..127, A stages of 32
// columns at 128 + 32 s
constexpr uint32_t kTmemAF8 = 128;
static_assert(kTmemAF8 + 32 * kStages <= kTmemCols, "TMEM budget (e4m3)");

struct MmaArgs {
    CUtensorMap tmW;        // packed weights [N][K/2] uint8, box 128 bytes x 128 rows
    const uint8_t* codes;   // activation tiles [nkb][BN][64] bf16, pre-swizzled
    const float* sw;        // [N]
    const float* sa;        // [M]
    float* Y;               // [M][N]
    int32_t* acc_out;       // optional [M][N]
    int32_t* part;          // [tiles][P][M][128] int32 piece slices when 1 < P <= kSliceMaxP
    int32_t* acc;           // [tiles][M][128] int32 accumulators when P > kSliceMaxP (zero between calls)
    unsigned* tickets;      // [tiles] when P > 1, zero between calls
    // group scales: sg [N][gld] fp32, gkb K blocks per group; with P > 1 the
    // fold's chunk sums go to part_f [tiles][nch][M][128] (chunks of
    // max(gkb, 16) K blocks)
    const float* sg;
    float* part_f;
    int gld, gkb, nch;
    int M, N, K, BN, P, nkb, kbp;
    // e4m3 path: the activation pass's per-piece code sums [M][pre_pieces]
    const int32_t* sum_part;
    int pre_pieces;
};

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
        #pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            atomicOr(&g_mma_error, kErrFullWait);
            return false;
        }
    }
}

// Waits (bounded, ignoring the abort flag) for a copy this thread issued,
// so that nothing lands in shared memory after the CTA exits.
__device__ __forceinline__ void drain(uint32_t bar, uint32_t parity) {
    if (!mbar_wait(bar, parity)) atomicOr(&g_mma_error, kErrDrainWait);
}

// Activation codes for the tensor cores, in the order the MMA reads them:
// K-block kb (64 codes of every row) is one contiguous [BN][64] bf16 tile of
// BN * 128 bytes, already in the 128-byte swizzled layout (16-byte chunk c
// of row m at m * 128 + ((c ^ (m % 8)) * 16)), so one 1-D bulk copy moves
// a whole tile.  Rows M..BN-1 and codes past K are zero.  Grid (BN rows,
// pieces of 256 vectors of 8 codes): every CTA of a row takes the row's
// max|x| (exact in binary16), s_a = max/127 by IEEE division, and quantizes
// its piece with the fast exact quantizer (actq.cuh); when X is null it
// widens the given int8 codes Xq instead.  Optional int8 codes and scale
// outputs for the caller.  It also zeroes the int32 accumulators of the
// atomic split plans that follow (acc_words of them).
__global__ void __launch_bounds__(kAQThreads) act_codes_kernel(
    const __half* __restrict__ X, const int8_t* __restrict__ Xq, const float* __restrict__ sa_in,
    int M, int64_t K, int BN, uint8_t* __restrict__ B, float* __restrict__ sa_ws,
    int8_t* __restrict__ Xq_out, float* __restrict__ sa_out, int32_t* __restrict__ acc,
    int64_t acc_words) {
    __shared__ float red[kAQThreads / 32];
    griddep_launch_dependents();
    griddep_wait();
    for (int64_t e = ((int64_t)blockIdx.y * gridDim.x + blockIdx.x) * kAQThreads + threadIdx.x; e < acc_words;
         e += (int64_t)gridDim.x * gridDim.y * kAQThreads)
        acc[e] = 0;
    const int m = blockIdx.x;
    const int64_t u = (int64_t)blockIdx.y * kAQThreads + threadIdx.x;  // vector of 8 codes
    const int64_t nchunks = (K + kKBlock - 1) / kKBlock * 8;           // incl. the padding to a K block
    const int64_t kchunks = K / 8;
    uint4* dst = reinterpret_cast<uint4*>(B + (u >> 3) * ((size_t)BN * 128) + (size_t)m * 128 +
                                          ((((int)u & 7) ^ (m & 7)) << 4));
    if (m >= M) {
        if (u < nchunks) *dst = make_uint4(0u, 0u, 0u, 0u);
        return;
    }
    float s;
    const uint4* xv = reinterpret_cast<const uint4*>(X + (int64_t)m * K);
    if (X == nullptr) {
        s = sa_in[m];
    } else {
        __half2 hm = __float2half2_rn(0.f);
        #pragma unroll 4
        for (int64_t v = threadIdx.x; v < kchunks; v += kAQThreads) {
            const uint4 h = xv[v];
            const __half2* p2 = reinterpret_cast<const __half2*>(&h);
            #pragma unroll
            for (int t = 0; t < 4; ++t) hm = __hmax2(hm, __habs2(p2[t]));
        }
        float mx = fmaxf(__low2float(hm), __high2float(hm));
        #pragma unroll
        for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
        __syncthreads();
        mx = 0.f;
        #pragma unroll
        for (int w = 0; w < kAQThreads / 32; ++w) mx = fmaxf(mx, red[w]);
        s = __fdiv_rn(mx, 127.f);
    }
    if (u < nchunks) {
        uint32_t o[4] = {0u, 0u, 0u, 0u};
        if (u < kchunks) {
            uint32_t c8[2];
            if (X != nullptr) {
                float r_lo, r_hi;
                quant_bracket(s, &r_lo, &r_hi);
                const uint2 q = quant8_split(xv[u], s, r_lo, r_hi);  // even / odd codes
                c8[0] = __byte_perm(q.x, q.y, 0x5140);               // natural order
                c8[1] = __byte_perm(q.x, q.y, 0x7362);
                if (Xq_out != nullptr)
                    *reinterpret_cast<uint2*>(Xq_out + (int64_t)m * K + 8 * u) = make_uint2(c8[0], c8[1]);
            } else {
                const uint2 c = *reinterpret_cast<const uint2*>(Xq + (int64_t)m * K + 8 * u);
                c8[0] = c.x;
                c8[1] = c.y;
            }
            // binary16 pairs in the permuted K order of the weight
            // converters: pair t = codes (t, t + 4) of the 8
            #pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int lo = (int)(int8_t)((c8[0] >> (8 * t)) & 0xFFu);
                const int hi = (int)(int8_t)((c8[1] >> (8 * t)) & 0xFFu);
                const __half2 v = __floats2half2_rn((float)lo, (float)hi);
                o[t] = *reinterpret_cast<const uint32_t*>(&v);
            }
        }
        *dst = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (blockIdx.y == 0 && threadIdx.x == 0) {
        sa_ws[m] = s;
        if (sa_out != nullptr) sa_out[m] = s;
    }
}

// The same for the e4m3 operand path: an INT8 code a = 16 a_hi + a_lo with
// a_hi = a >> 4 in [-8, 7] and a_lo = a & 15 in [0, 15], both exact in
// e4m3.  Per 128-code K tile t the B operand is [2 BN][128] bytes at
// t * 2 BN * 128: rows 0..BN-1 hold a_hi of the batch rows, BN..2BN-1 a_lo,
// 128-byte swizzled (16-byte chunk c of row m at m * 128 + (c ^ (m % 8)) * 16),
// each group of 8 codes in the order (0, 2, 4, 6, 1, 3, 5, 7) that the
// weight converters produce.  One MMA then yields W.A_hi and W.A_lo side by
// side in D.  Thread u handles 16 codes (one chunk); each CTA also writes the
// exact sum of its piece's codes of row m (sum_part[m][piece]), which removes
// the +8 bias of the weight encoding.
__device__ __forceinline__ uint32_t e4m3x4(int v0, int v1, int v2, int v3) {
    return (uint32_t)__nv_cvt_float_to_fp8((float)v0, __NV_SATFINITE, __NV_E4M3) |
           ((uint32_t)__nv_cvt_float_to_fp8((float)v1, __NV_SATFINITE, __NV_E4M3) << 8) |
           ((uint32_t)__nv_cvt_float_to_fp8((float)v2, __NV_SATFINITE, __NV_E4M3) << 16) |
           ((uint32_t)__nv_cvt_float_to_fp8((float)v3, __NV_SATFINITE, __NV_E4M3) << 24);
}

__global__ void __launch_bounds__(kAQThreads) act_codes_e4m3_kernel(
    const __half* __restrict__ X, const int8_t* __restrict__ Xq, const float* __restrict__ sa_in,
    int M, int64_t K, int BN, uint8_t* __restrict__ B, float* __restrict__ sa_ws,
    int8_t* __restrict__ Xq_out, float* __restrict__ sa_out, int32_t* __restrict__ acc,
    int64_t acc_words, int32_t* __restrict__ sum_part) {
    __shared__ float red[kAQThreads / 32];
    __shared__ int isum[kAQThreads / 32];
    griddep_launch_dependents();
    griddep_wait();
    for (int64_t e = ((int64_t)blockIdx.y * gridDim.x + blockIdx.x) * kAQThreads + threadIdx.x; e < acc_words;
         e += (int64_t)gridDim.x * gridDim.y * kAQThreads)
        acc[e] = 0;
    const int m = blockIdx.x;
    const int64_t u = (int64_t)blockIdx.y * kAQThreads + threadIdx.x;  // chunk of 16 codes
    const int64_t nchunks = (K + 127) / 128 * 8;                        // incl. the padding to a K tile
    const int64_t kchunks = K / 16;                                      // K % 32 == 0
    const int64_t t = u >> 3;
    const int c = (int)(u & 7);
    const size_t tile = (size_t)t * 2 * BN * 128;
    uint4* dhi = reinterpret_cast<uint4*>(B + tile + (size_t)m * 128 + ((c ^ (m & 7)) << 4));
    const int ml = BN + m;
    uint4* dlo = reinterpret_cast<uint4*>(B + tile + (size_t)ml * 128 + ((c ^ (ml & 7)) << 4));
    if (m >= M) {
        if (u < nchunks) *dhi = *dlo = make_uint4(0u, 0u, 0u, 0u);
        return;
    }
    float s;
    const uint4* xv = reinterpret_cast<const uint4*>(X + (int64_t)m * K);
    if (X == nullptr) {
        s = sa_in[m];
    } else {
        __half2 hm = __float2half2_rn(0.f);
        #pragma unroll 4
        for (int64_t v = threadIdx.x; v < K / 8; v += kAQThreads) {
            const uint4 h = xv[v];
            const __half2* p2 = reinterpret_cast<const __half2*>(&h);
            #pragma unroll
            for (int q = 0; q < 4; ++q) hm = __hmax2(hm, __habs2(p2[q]));
        }
        float mx = fmaxf(__low2float(hm), __high2float(hm));
        #pragma unroll
        for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
        __syncthreads();
        mx = 0.f;
        #pragma unroll
        for (int w = 0; w < kAQThreads / 32; ++w) mx = fmaxf(mx, red[w]);
        s = __fdiv_rn(mx, 127.f);
    }
    int rsum = 0;
    if (u < nchunks) {
        uint4 hi = make_uint4(0u, 0u, 0u, 0u), lo = hi;
        if (u < kchunks) {
            uint32_t c8[4];  // the 16 codes in natural order
            if (X != nullptr) {
                float r_lo, r_hi;
                quant_bracket(s, &r_lo, &r_hi);
                #pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint2 q = quant8_split(xv[2 * u + h], s, r_lo, r_hi);  // even / odd codes
                    c8[2 * h] = __byte_perm(q.x, q.y, 0x5140);
                    c8[2 * h + 1] = __byte_perm(q.x, q.y, 0x7362);
                }
                if (Xq_out != nullptr)
                    *reinterpret_cast<uint4*>(Xq_out + (int64_t)m * K + 16 * u) =
                        make_uint4(c8[0], c8[1], c8[2], c8[3]);
            } else {
                const uint4 cq = *reinterpret_cast<const uint4*>(Xq + (int64_t)m * K + 16 * u);
                c8[0] = cq.x;
                c8[1] = cq.y;
                c8[2] = cq.z;
                c8[3] = cq.w;
            }
            // each 8-code group in the converters' order (0, 2, 4, 6, 1, 3, 5, 7)
            const uint32_t p8[4] = {__byte_perm(c8[0], c8[1], 0x6420), __byte_perm(c8[0], c8[1], 0x7531),
                                    __byte_perm(c8[2], c8[3], 0x6420), __byte_perm(c8[2], c8[3], 0x7531)};
            uint32_t h4[4], l4[4];
            #pragma unroll
            for (int w = 0; w < 4; ++w) {
                int a[4];
                #pragma unroll
                for (int b = 0; b < 4; ++b) {
                    a[b] = (int)(int8_t)((p8[w] >> (8 * b)) & 0xFFu);
                    rsum += a[b];
                }
                h4[w] = e4m3x4(a[0] >> 4, a[1] >> 4, a[2] >> 4, a[3] >> 4);
                l4[w] = e4m3x4(a[0] & 15, a[1] & 15, a[2] & 15, a[3] & 15);
            }
            hi = make_uint4(h4[0], h4[1], h4[2], h4[3]);
            lo = make_uint4(l4[0], l4[1], l4[2], l4[3]);
        }
        *dhi = hi;
        *dlo = lo;
    }
    // the piece's exact sum of codes (|sum| <= 127 * 4096)
    #pragma unroll
    for (int o = 16; o >= 1; o >>= 1) rsum += __shfl_xor_sync(0xFFFFFFFFu, rsum, o);
    if ((threadIdx.x & 31) == 0) isum[threadIdx.x >> 5] = rsum;
    __syncthreads();
    if (threadIdx.x == 0) {
        int tsum = 0;
        #pragma unroll
        for (int w = 0; w < kAQThreads / 32; ++w) tsum += isum[w];
        sum_part[(int64_t)m * gridDim.y + blockIdx.y] = tsum;
    }
    if (blockIdx.y == 0 && threadIdx.x == 0) {
        sa_ws[m] = s;
        if (sa_out != nullptr) sa_out[m] = s;
    }
}

// One packed word (8 INT4 codes, low nibble first) -> 8 binary16 values in
// the permuted K order (t, t + 4) per 32-bit pair, t = 0..3, the order the
// activation tiles use too (a fixed permutation of K inside each 8-code
// group leaves the dot product unchanged).  Nibbles 0 and 4 masked in place
// and xor'ed into the mantissa of 1024.0 give 1024 + (n ^ 8) = 1032 + q;
// nibbles 1 and 5 masked in place give 1024 + 16 (q + 8), scaled by 1/16
// with one fma; the word shifted by 8 gives nibbles 2, 6 and 3, 7.  Every
// step is exact: 4 mask-xor, 1 shift and 4 half2 operations per 8 codes.
__device__ __forceinline__ uint4 int4x8_to_f16(uint32_t w) {
    const uint32_t w2 = w >> 8;
    const uint32_t x0 = (w & 0x000F000Fu) ^ 0x64086408u;   // codes 0, 4: 1032 + q
    const uint32_t x1 = (w & 0x00F000F0u) ^ 0x64806480u;   // codes 1, 5: 1024 + 16 (q + 8)
    const uint32_t x2 = (w2 & 0x000F000Fu) ^ 0x64086408u;  // codes 2, 6
    const uint32_t x3 = (w2 & 0x00F000F0u) ^ 0x64806480u;  // codes 3, 7
    const __half2 b0 = __floats2half2_rn(1032.f, 1032.f);
    const __half2 s1 = __floats2half2_rn(0.0625f, 0.0625f);
    const __half2 b1 = __floats2half2_rn(-72.f, -72.f);
    const __half2 v0 = __hsub2(*reinterpret_cast<const __half2*>(&x0), b0);
    const __half2 v1 = __hfma2(*reinterpret_cast<const __half2*>(&x1), s1, b1);
    const __half2 v2 = __hsub2(*reinterpret_cast<const __half2*>(&x2), b0);
    const __half2 v3 = __hfma2(*reinterpret_cast<const __half2*>(&x3), s1, b1);
    return make_uint4(*reinterpret_cast<const uint32_t*>(&v0), *reinterpret_cast<const uint32_t*>(&v1),
                      *reinterpret_cast<const uint32_t*>(&v2), *reinterpret_cast<const uint32_t*>(&v3));
}

// One packed word (8 INT4 codes) -> 8 e4m3 bytes in the K order (0, 2, 4, 6,
// 1, 3, 5, 7): code q becomes the byte v = n ^ 8 = q + 8 in [0, 15], which as
// e4m3 is exactly v * 2^-9 (bytes 0..7 are the subnormals m * 2^-9, bytes
// 8..15 the first binade (8 + m) * 2^-9).  One xor, one shift, two masks.
__device__ __forceinline__ uint2 int4x8_to_e4m3(uint32_t w) {
    const uint32_t x = w ^ 0x88888888u;
    return make_uint2(x & 0x0F0F0F0Fu, (x >> 4) & 0x0F0F0F0Fu);
}

// Two CTAs per SM (shared memory < 113 KB, 256 TMEM columns, <= 93
// registers): the SM's tensor core then interleaves two MMA streams, each at
// the issue rate of one.
//
// kG: group-wise weight scales (groups of gkb K blocks, a whole number of
// stages; K pieces of whole fold chunks).  The MMAs of each group start a
// fresh accumulator D (exact integer sums); when a group's last stage is
// committed (dfull), every converter warp folds its share of D in the fixed
// order of the group-scale contract: inside each chunk of max(group, 1024)
// codes f = fma(D, s_g, f) with f in TMEM (F, +0 at the chunk's first
// group), and at the chunk's last group T = T + f into the thread's
// registers (one piece: Y = T * s_a at the end), or f to the workspace
// (split K: the CTA that finishes a tile last adds the chunks in order).
// Then it releases D (dfree) for the next group.  A converter warp does the readout of a group before it
// converts the stage `lag` stages past the group's end, so every wait
// points at earlier work.
//
// kF8 (row-wise scales only): the e4m3 operand path.  Weight codes are
// widened to e4m3 (four per TMEM column, a stage of 128 codes in 32
// columns), the activation tiles hold a_hi and a_lo as 2 BN rows, and each
// MMA (kind::f8f6f4, K = 32) covers twice the weights of a kind::f16 MMA;
// D holds W.A_hi in columns 0..BN-1 and W.A_lo in BN..2BN-1, both exact
// integers in fp32, and acc = 16 D_hi + D_lo.
// kAtomic (row-wise plans with more than kSliceMaxP K pieces): the atomic
// split epilogue, compiled apart so that the register-held epilogue of the
// other plans does not raise this variant's register allocation.
template <bool kG, bool kF8, bool kAtomic>
__global__ void __launch_bounds__(kMmaThreads, 2) mma_kernel(const __grid_constant__ MmaArgs a) {
    static_assert(!(kG && kF8), "the e4m3 path has row-wise scales only");
    static_assert(!(kG && kAtomic), "group scales add their chunk sums in order");
    constexpr int S = kG ? kStagesG : kStages;          // stage ring in use
    constexpr uint32_t kA0 = kF8 ? kTmemAF8 : kG ? kTmemAG : kTmemA;  // first A stage column
    constexpr uint32_t kAStage = kF8 ? 32 : kTmemAStage;               // A columns per stage
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base for the swizzled tiles
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sbase = smem_u32(smem);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int tile = blockIdx.x / a.P;
    const int p = blockIdx.x % a.P;
    const int n0 = tile * kTileRows;
    const int kb0 = p * a.kbp;
    const int nk = min(a.nkb, kb0 + a.kbp) - kb0;  // >= 1 by the plan
    const int BN = a.BN;
    const uint32_t b_bytes = (uint32_t)BN * kKBlock * 2;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
    uint64_t* wfull = bars;
    uint64_t* wempty = wfull + kWStages;
    uint64_t* afull = wempty + kWStages;  // A stage written (4 converter warps)
    uint64_t* bfull = afull + kStages;    // B stage landed
    uint64_t* sempty = bfull + kStages;   // stage consumed by the MMAs (commit)
    uint64_t* accfull = sempty + kStages;
    uint64_t* dfull = accfull + 1;        // group scales [buffer]: a group's sums are in D
    uint64_t* dfree = dfull + 2;          // group scales [buffer]: every converter warp has read D
    const int nst = (nk + kStageK - 1) / kStageK;  // stages of this piece
    const int spg = kG ? a.gkb / kStageK : 1;      // stages per group
    // group g uses D buffer g % nbuf (columns 32 (g % nbuf)); buffer b
    // completes dfull[b] / dfree[b] phase g / nbuf.  The converter warps read
    // group g out before converting stage last(g) + lag: with two buffers a
    // stage later, so that a conversion never waits for the MMAs of the stage
    // just before it (the next group's MMAs wait only for the readout of the
    // group before the previous one).
    const int nbuf = (kG && BN <= 32) ? 2 : 1;
    const int lag = nbuf;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
    int* last_flag = reinterpret_cast<int*>(smem + kOffMisc + 8);
    const uint32_t ncols = kTmemCols;  // half of the SM's 512: two CTAs per SM

    if (tid == 0) {
        for (int s = 0; s < kWStages; ++s) {
            mbar_init(smem_u32(wfull + s), 1);
            mbar_init(smem_u32(wempty + s), 4 * (kWBlocks / kStageK));  // each stage read by 4 warps
        }
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(afull + s), 4);  // the 4 lane quarters of one group
            mbar_init(smem_u32(bfull + s), 1);
            mbar_init(smem_u32(sempty + s), 1);
        }
        mbar_init(smem_u32(accfull), 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(dfull + b), 1);
            mbar_init(smem_u32(dfree + b), kConvWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), ncols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    griddep_launch_dependents();

    if (warp == 0) {
        // ---- producer: packed INT4 tiles (weights may be read before the
        // dependency wait)
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            int issued = 0;
            const int nw = (nk + kWBlocks - 1) / kWBlocks;  // loads of kWBlocks K blocks each
            for (int i = 0; i < nw; ++i) {
                const int s = i % kWStages;
                if (i >= kWStages && !wait_bounded(smem_u32(wempty + s), ((i / kWStages) - 1) & 1, abort_flag))
                    break;
                mbar_arrive_expect_tx(smem_u32(wfull + s), kWTileBytes);
                tma_load_2d_hint(sbase + kOffW + s * kWTileBytes, &a.tmW, (kb0 + kWBlocks * i) * (kKBlock / 2),
                                 n0, smem_u32(wfull + s), pol);
                issued = i + 1;
            }
            for (int i = max(0, issued - kWStages); i < issued; ++i)
                drain(smem_u32(wfull + i % kWStages), (i / kWStages) & 1);
        }
    } else if (warp == 1) {
        // ---- MMA issuer (one lane): per stage up to kStageK K blocks of
        // four K = 16 steps, then one commit that frees the stage
        if (lane == 0) {
            const uint32_t idesc = kF8 ? e4m3_idesc(kTileRows, 2 * BN) : f16_idesc(kTileRows, BN);
            for (int st = 0; st < nst; ++st) {
                const int s = st % S;
                const uint32_t ph = (st / S) & 1;
                // group scales: a group's first stage starts D afresh, once
                // the converter warps have read the previous group's sums
                const bool first = kG && (st % spg) == 0;
                const int g = kG ? st / spg : 0;
                if (first && g >= nbuf &&
                    !wait_bounded(smem_u32(dfree + g % nbuf), ((g / nbuf) - 1) & 1, abort_flag))
                    break;
                const uint32_t d_tmem = tmem + (uint32_t)(32 * (g % nbuf));
                if (!wait_bounded(smem_u32(afull + s), ph, abort_flag)) break;
                if (!wait_bounded(smem_u32(bfull + s), ph, abort_flag)) break;
                tc_fence_after_sync();
                const int nkb = min(kStageK, nk - kStageK * st);
                const uint32_t at = tmem + kA0 + kAStage * s;
                if constexpr (kF8) {
                    // one [2 BN][128] e4m3 tile a stage (zero past K): four K = 32 steps
                    const uint64_t bd = sw128_desc(sbase + kOffB + s * kBStageMax);
                    #pragma unroll
                    for (int k = 0; k < 4; ++k)
                        tc_mma_e4m3_tmem_a(d_tmem, at + 8 * k, bd + 2 * k, idesc, st > 0 || k > 0);
                }
                for (int j = 0; j < (kF8 ? 0 : nkb); ++j) {
                    const uint64_t bd = sw128_desc(sbase + kOffB + s * kBStageMax + j * b_bytes);
                    #pragma unroll
                    for (int k = 0; k < kKBlock / 16; ++k) {  // 8 TMEM columns of A, 32 bytes of B a step
                        const bool acc = kG ? !(first && j == 0 && k == 0) : (st > 0 || j > 0 || k > 0);
                        tc_mma_f16_tmem_a(d_tmem, at + 32 * j + 8 * k, bd + 2 * k, idesc, acc);
                    }
                }
                tc_commit(smem_u32(sempty + s));
                if (kG && (st % spg) == spg - 1) tc_commit(smem_u32(dfull + g % nbuf));  // the group's D is complete
            }
            tc_commit(smem_u32(accfull));  // every MMA issued so far
        }
    } else if (warp == 2) {
        // ---- activation tiles (one lane): the K blocks of a stage are
        // adjacent in the tiled codes, one bulk copy each
        if (lane == 0) {
            griddep_wait();  // the bf16 codes come from the previous kernel
            const uint64_t pol = l2_evict_last_policy();
            int issued = 0;
            for (int st = 0; st < nst; ++st) {
                const int s = st % S;
                if (st >= S && !wait_bounded(smem_u32(sempty + s), ((st / S) - 1) & 1, abort_flag))
                    break;
                const uint32_t bytes = kF8 ? (uint32_t)kStageK * b_bytes
                                           : (uint32_t)min(kStageK, nk - kStageK * st) * b_bytes;
                mbar_arrive_expect_tx(smem_u32(bfull + s), bytes);
                bulk_g2s(sbase + kOffB + s * kBStageMax, a.codes + (size_t)(kb0 + kStageK * st) * b_bytes,
                         bytes, smem_u32(bfull + s), pol);
                issued = st + 1;
            }
            for (int st = max(0, issued - S); st < issued; ++st)
                drain(smem_u32(bfull + st % S), (st / S) & 1);
        }
    } else {
        // ---- converters: each thread widens its weight row's 64 codes of a
        // stage to bf16 and stores them into the stage's TMEM columns (the
        // MMA's A operand); the two groups take alternate stages
        const int cg = (warp - kFirstConvWarp) >> 2;
        const int q = warp & 3;         // TMEM lanes 32q .. 32q + 31
        const int r = 32 * q + lane;    // weight row within the tile
        const uint32_t lanes = tmem + ((uint32_t)(32 * q) << 16);
        // group scales: fold group g's sums (this warp's lanes, its column
        // chunks ch = cg + 2j) into the chunk sum f in TMEM, and at a chunk's
        // last group into the totals T; false when a wait gave up
        int next_g = 0;
        const int ngroups = kG ? nst / spg : 0;
        const int gpc = kG ? max(1, 16 / a.gkb) : 1;  // groups per 1024-code (or one-group) chunk
        float T[kG ? 4 : 1][8];
        #pragma unroll
        for (int j = 0; j < (kG ? 4 : 1); ++j)
            #pragma unroll
            for (int t = 0; t < 8; ++t) T[j][t] = 0.f;
        const int g0 = kG ? kb0 / a.gkb : 0;  // first group of the piece (a chunk's first)
        auto readout = [&](int gl) -> bool {
            const int n = n0 + r;
            const int g = g0 + gl;  // group index in the row
            const float sc = n < a.N ? __ldg(a.sg + (int64_t)n * a.gld + g) : 0.f;
            const int b = gl % nbuf;
            if (!__all_sync(0xFFFFFFFFu, wait_bounded(smem_u32(dfull + b), (gl / nbuf) & 1, abort_flag)))
                return false;
            tc_fence_after_sync();
            const bool cfirst = (g % gpc) == 0;
            const bool clast = (g % gpc) == gpc - 1 || gl == ngroups - 1;
            #pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int ch = cg + kConvGroups * j;
                if (ch < BN / 8) {
                    uint32_t d[8], f[8];
                    tmem_ld8(lanes + (uint32_t)(32 * b + 8 * ch), d);
                    if (!cfirst) {
                        tmem_ld8(lanes + kTmemF + (uint32_t)(8 * ch), f);
                    } else {
                        #pragma unroll
                        for (int t = 0; t < 8; ++t) f[t] = 0u;
                    }
                    #pragma unroll
                    for (int t = 0; t < 8; ++t)  // D holds an exact integer
                        f[t] = __float_as_uint(__fmaf_rn(__uint_as_float(d[t]), sc, __uint_as_float(f[t])));
                    if (clast && a.P == 1) {
                        #pragma unroll
                        for (int t = 0; t < 8; ++t) T[kG ? j : 0][t] = __fadd_rn(T[kG ? j : 0][t], __uint_as_float(f[t]));
                    } else if (clast) {
                        float* dst = a.part_f + ((int64_t)(tile * a.nch + g / gpc) * a.M) * kTileRows + r;
                        #pragma unroll
                        for (int t = 0; t < 8; ++t)
                            if (8 * ch + t < a.M) dst[(int64_t)(8 * ch + t) * kTileRows] = __uint_as_float(f[t]);
                    } else {
                        tmem_st8(lanes + kTmemF + (uint32_t)(8 * ch), f);
                    }
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(dfree + b));
            return true;
        };
        for (int st = cg; st < nst; st += kConvGroups) {
            if constexpr (kG) {  // groups that end before this stage
                bool alive = true;
                while (alive && next_g < ngroups && (next_g + 1) * spg - 1 + lag <= st) {
                    alive = readout(next_g);
                    if (alive) ++next_g;
                }
                if (!alive) break;
            }
            const int kb = kStageK * st;  // first K block of the stage (within the piece)
            const int t = kb / kWBlocks, sub = kb % kWBlocks;
            const int ws = t % kWStages;
            // warp-uniform outcome: a lane may time out while another sees the phase
            if (!__all_sync(0xFFFFFFFFu, wait_bounded(smem_u32(wfull + ws), (t / kWStages) & 1, abort_flag)))
                break;
            // 128-byte rows swizzled by the TMA: 16-byte chunk c of row r at (c ^ r % 8) * 16;
            // K block sub + j of the load is chunks 2(sub + j) and 2(sub + j) + 1
            const uint8_t* row = smem + kOffW + ws * kWTileBytes + r * 128;
            uint4 c16[2 * kStageK];
            #pragma unroll
            for (int c = 0; c < 2 * kStageK; ++c)
                c16[c] = *reinterpret_cast<const uint4*>(row + (((2 * sub + c) ^ (r & 7)) << 4));
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(wempty + ws));
            const int s = st % S;
            if (st >= S &&
                !__all_sync(0xFFFFFFFFu, wait_bounded(smem_u32(sempty + s), ((st / S) - 1) & 1, abort_flag)))
                break;
            if constexpr (kF8) {  // word w of K block j = codes 64 j + 8 w .. + 7 -> columns 16 j + 2 w, + 1
                uint32_t v[32];
                #pragma unroll
                for (int j = 0; j < kStageK; ++j) {
                    const uint32_t w8[8] = {c16[2 * j].x, c16[2 * j].y, c16[2 * j].z, c16[2 * j].w,
                                            c16[2 * j + 1].x, c16[2 * j + 1].y, c16[2 * j + 1].z, c16[2 * j + 1].w};
                    #pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        const uint2 o = int4x8_to_e4m3(w8[w]);
                        v[16 * j + 2 * w] = o.x;
                        v[16 * j + 2 * w + 1] = o.y;
                    }
                }
                tmem_st32(lanes + kA0 + kAStage * s, v);
            }
            #pragma unroll
            for (int j = 0; j < (kF8 ? 0 : kStageK); ++j) {  // word w of K block j = codes 8w .. 8w+7 -> columns 4w .. 4w+3
                const uint32_t w8[8] = {c16[2 * j].x, c16[2 * j].y, c16[2 * j].z, c16[2 * j].w,
                                        c16[2 * j + 1].x, c16[2 * j + 1].y, c16[2 * j + 1].z, c16[2 * j + 1].w};
                uint32_t v[32];
                #pragma unroll
                for (int w = 0; w < 8; ++w) {
                    const uint4 o = int4x8_to_f16(w8[w]);
                    v[4 * w] = o.x;
                    v[4 * w + 1] = o.y;
                    v[4 * w + 2] = o.z;
                    v[4 * w + 3] = o.w;
                }
                tmem_st32(lanes + kA0 + kAStage * s + 32 * j, v);
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(afull + s));
        }

        if constexpr (kG) {
            // ---- epilogue, group scales: the remaining groups, then
            // Y = T * s_a
            while (next_g < ngroups && readout(next_g)) ++next_g;
            griddep_wait();  // activation scales and outputs
            const bool ok = __all_sync(0xFFFFFFFFu, next_g == ngroups);
            tc_fence_after_sync();
            const int n = n0 + r;
            if (a.P == 1) {
                if (ok && n < a.N) {
                    #pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int ch = cg + kConvGroups * j;
                        if (ch < BN / 8) {
                            #pragma unroll
                            for (int t = 0; t < 8; ++t) {
                                const int m = 8 * ch + t;
                                if (m < a.M) a.Y[(int64_t)m * a.N + n] = __fmul_rn(T[j][t], a.sa[m]);
                            }
                        }
                    }
                }
            } else {
                // the last CTA of the tile adds the chunk sums in chunk order;
                // every converter warp meets at the barrier, and after a wait
                // gave up (the CTA's abort flag) nothing is written
                const int ct = tid - kFirstConvWarp * 32;
                __threadfence();
                named_bar_sync(1, kConvWarps * 32);
                if (ct == 0) *last_flag = !*abort_flag && (atomicAdd(a.tickets + tile, 1u) == (unsigned)(a.P - 1));
                named_bar_sync(1, kConvWarps * 32);
                if (*last_flag) {
                    __threadfence();
                    const int rows = min(kTileRows, a.N - n0);
                    for (int e = ct; e < a.M * kTileRows; e += kConvWarps * 32) {
                        const int m = e / kTileRows, rr = e % kTileRows;
                        if (rr >= rows) continue;
                        const float* src = a.part_f + ((int64_t)tile * a.nch * a.M + m) * kTileRows + rr;
                        // chunk order; loads issued 8 at a time ahead of the adds
                        float t = 0.f;
                        for (int c0 = 0; c0 < a.nch; c0 += 8) {
                            float v[8];
                            #pragma unroll
                            for (int k = 0; k < 8; ++k)
                                v[k] = c0 + k < a.nch ? __ldcg(src + (int64_t)(c0 + k) * a.M * kTileRows) : 0.f;
                            #pragma unroll
                            for (int k = 0; k < 8; ++k)
                                if (c0 + k < a.nch) t = __fadd_rn(t, v[k]);
                        }
                        a.Y[(int64_t)m * a.N + n0 + rr] = __fmul_rn(t, a.sa[m]);
                    }
                    if (ct == 0) a.tickets[tile] = 0u;  // ready for the next call
                }
            }
        } else {
            // ---- epilogue: TMEM lanes = weight rows, columns = batch rows
            griddep_wait();  // scales and outputs
            const int ct = tid - kFirstConvWarp * 32;
            int* sa_sum = reinterpret_cast<int*>(smem + kOffSaSum);
            if constexpr (kF8) {
                // the batch rows' exact code sums (the +8 bias of the weight bytes)
                for (int e = ct; e < a.M; e += kConvWarps * 32) sa_sum[e] = 0;
                named_bar_sync(1, kConvWarps * 32);
                for (int e = ct; e < a.M * a.pre_pieces; e += kConvWarps * 32)
                    atomicAdd(sa_sum + e / a.pre_pieces, __ldcg(a.sum_part + e));
                named_bar_sync(1, kConvWarps * 32);
            }
            const bool ok = __all_sync(0xFFFFFFFFu, wait_bounded(smem_u32(accfull), 0, abort_flag));
            tc_fence_after_sync();
            // the TMEM lanes this warp may read are its converter lanes (q, r);
            // the two warps of a quarter split the columns: ch = cg + 2j
            const int n = n0 + r;
            const float swv = (ok && n < a.N) ? a.sw[n] : 0.f;
            // e4m3: D = 2^-9 sum v b (weight bytes v = q + 8), so 512 D is an
            // exact integer and sum q a = 16 U_hi + U_lo - 8 sum a
            auto exact_sum = [&](uint32_t v, uint32_t vl) -> int32_t {
                return kF8 ? 16 * __float2int_rn(__uint_as_float(v) * 512.f) + __float2int_rn(__uint_as_float(vl) * 512.f)
                           : __float2int_rn(__uint_as_float(v));
            };
            auto rescale = [&](int m, int64_t o, int32_t raw, float swn) {
                const int32_t acc = kF8 ? raw - 8 * sa_sum[m] : raw;
                a.Y[o] = __fmul_rn(__fmul_rn(__int2float_rn(acc), swn), a.sa[m]);
                if (a.acc_out != nullptr) a.acc_out[o] = acc;
            };
            if constexpr (kAtomic) {
                // split K into many pieces: every piece adds its sums into the
                // tile's int32 accumulator [M][128] (integer addition: exact,
                // order-free; the reduction spread over every CTA); the last
                // CTA rescales the totals and clears them for the next matrix
                // or call.  Every converter warp meets at the barrier.
                int32_t* acc_t = a.acc + (int64_t)tile * a.M * kTileRows;
                for (int ch = cg; ch < BN / 8; ch += kConvGroups) {
                    uint32_t v[8], vl[8];
                    tmem_ld8(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(8 * ch), v);
                    if constexpr (kF8) tmem_ld8(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(BN + 8 * ch), vl);
                    if (!ok) continue;
                    #pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        const int m = 8 * ch + t;
                        if (m >= a.M) break;
                        atomicAdd(acc_t + (int64_t)m * kTileRows + r, exact_sum(v[t], vl[t]));
                    }
                }
                __threadfence();
                named_bar_sync(1, kConvWarps * 32);
                if (ct == 0) *last_flag = !*abort_flag && (atomicAdd(a.tickets + tile, 1u) == (unsigned)(a.P - 1));
                named_bar_sync(1, kConvWarps * 32);
                if (*last_flag) {
                    __threadfence();
                    const int rows = min(kTileRows, a.N - n0);
                    constexpr int kBatch = 8;  // loads in flight per thread
                    for (int e0 = ct; e0 < a.M * kTileRows; e0 += kConvWarps * 32 * kBatch) {
                        int32_t v[kBatch];
                        #pragma unroll
                        for (int b = 0; b < kBatch; ++b) {
                            const int e = e0 + b * kConvWarps * 32;
                            v[b] = e < a.M * kTileRows ? __ldcg(acc_t + e) : 0;
                        }
                        #pragma unroll
                        for (int b = 0; b < kBatch; ++b) {
                            const int e = e0 + b * kConvWarps * 32;
                            if (e >= a.M * kTileRows) break;
                            __stcg(acc_t + e, 0);
                            const int m = e / kTileRows, rr = e % kTileRows, nn = n0 + rr;
                            if (rr < rows) rescale(m, (int64_t)m * a.N + nn, v[b], a.sw[nn]);
                        }
                    }
                    if (ct == 0) a.tickets[tile] = 0u;  // ready for the next call
                }
            } else {
                int32_t raw[4][8];  // this thread's exact sums (e4m3: before the bias)
                #pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int ch = cg + kConvGroups * j;
                    #pragma unroll
                    for (int t = 0; t < 8; ++t) raw[j][t] = 0;
                    if (ch < BN / 8) {  // uniform over the warp
                        uint32_t v[8], vl[8];
                        tmem_ld8(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(8 * ch), v);
                        if constexpr (kF8) tmem_ld8(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(BN + 8 * ch), vl);
                        #pragma unroll
                        for (int t = 0; t < 8; ++t) raw[j][t] = exact_sum(v[t], vl[t]);
                    }
                }
                // the outputs of this thread's row and columns from its exact sums
                auto write_out = [&]() {
                    if (!ok || n >= a.N) return;
                    #pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        #pragma unroll
                        for (int t = 0; t < 8; ++t) {
                            const int m = 8 * (cg + kConvGroups * j) + t;
                            if (m < a.M) rescale(m, (int64_t)m * a.N + n, raw[j][t], swv);
                        }
                    }
                };
                if (a.P == 1) {
                    write_out();
                } else {
                    // split K into a few pieces: every piece stores its int32
                    // slice [M][128] with plain stores; the CTA that takes the
                    // tile's last ticket adds the other pieces' values to the
                    // sums it holds (integer addition: exact, order-free), each
                    // thread for its own outputs with all its loads of a piece
                    // in flight at once.  Every converter warp meets at the
                    // barrier.
                    int32_t* part_t = a.part + (int64_t)tile * a.P * a.M * kTileRows + r;
                    const int64_t slice = (int64_t)a.M * kTileRows;
                    if (ok) {
                        #pragma unroll
                        for (int j = 0; j < 4; ++j)
                            #pragma unroll
                            for (int t = 0; t < 8; ++t) {
                                const int m = 8 * (cg + kConvGroups * j) + t;
                                if (m < a.M) __stcg(part_t + p * slice + (int64_t)m * kTileRows, raw[j][t]);
                            }
                    }
                    __threadfence();
                    named_bar_sync(1, kConvWarps * 32);
                    if (ct == 0) *last_flag = !*abort_flag && (atomicAdd(a.tickets + tile, 1u) == (unsigned)(a.P - 1));
                    named_bar_sync(1, kConvWarps * 32);
                    if (*last_flag) {
                        __threadfence();
                        for (int pp = 0; pp < a.P; ++pp) {
                            if (pp == p) continue;
                            int32_t o[4][8];
                            #pragma unroll
                            for (int j = 0; j < 4; ++j)
                                #pragma unroll
                                for (int t = 0; t < 8; ++t) {
                                    const int m = 8 * (cg + kConvGroups * j) + t;
                                    o[j][t] = m < a.M ? __ldcg(part_t + pp * slice + (int64_t)m * kTileRows) : 0;
                                }
                            #pragma unroll
                            for (int j = 0; j < 4; ++j)
                                #pragma unroll
                                for (int t = 0; t < 8; ++t) raw[j][t] += o[j][t];
                        }
                        write_out();
                        if (ct == 0) a.tickets[tile] = 0u;  // ready for the next call
                    }
                }
            }
        }
    }

    // every MMA has completed (accfull) before TMEM is released
    if (tid == 32) drain(smem_u32(accfull), 0);
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, ncols);
    }
}

// --------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
               uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swz) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       unsigned flags, void** args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (flags & 1u) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

bool make_w4_tile_map(void* map, const uint8_t* Wq, int64_t K, int64_t N) {
    return encode_2d(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_UINT8, Wq, (uint64_t)(K / 2),
                     (uint64_t)N, (uint64_t)(K / 2), kWBlocks * kKBlock / 2, kTileRows,
                     CU_TENSOR_MAP_SWIZZLE_128B);
}

bool make_mma_plan(int M, int64_t K, int64_t N, int num_sms, MmaPlan* out, int gkb, int force_p) {
    if (M < 1 || M > 64 || K < 32 || K % 32 || N < 1 || N > 0x7FFFFFFF) return false;
    // group scales: groups of gkb K blocks, whole stages, each group's sums
    // exact in fp32 (at most 256 K blocks)
    if (gkb != 0 && (gkb < kStageK || gkb % kStageK || gkb > 256 || K % ((int64_t)gkb * kKBlock)))
        return false;
    MmaPlan pl = {};
    pl.BN = (M + 15) / 16 * 16;
    pl.tiles = (int)((N + kTileRows - 1) / kTileRows);
    pl.nkb = (int)((K + kKBlock - 1) / kKBlock);
    // split K when the tiles alone leave SMs idle; pieces of at most 256
    // K-blocks (16384) keep every fp32 partial sum exact
    int P = 1;
    const int slots = 2 * num_sms;  // resident CTAs
    if (pl.tiles < slots * 4 / 5) P = slots / pl.tiles;
    // a split pays a fixed tail (the partials, a ticket, the last CTA's
    // adds): for a second CTA per SM (at most 2 pieces) worth it only for
    // pieces of at least 16 K blocks (1024 codes), else of at least 8
    if (P > (P <= 2 ? pl.nkb / 16 : pl.nkb / 8)) P = P <= 2 ? pl.nkb / 16 : pl.nkb / 8;
    if (force_p > 0) P = force_p;
    if (P < 1) P = 1;
    // row-wise scales: pieces of at most 256 K blocks keep the integer sums
    // exact; group scales: each group's D is exact on its own, pieces hold
    // whole fold chunks (max(gkb, 16) K blocks), and a split writes one fp32
    // chunk sum per output and chunk, allowed up to kGroupPartBytes
    const int pmin = gkb ? 1 : (pl.nkb + 255) / 256;
    if (P < pmin) P = pmin;
    const int cb = gkb > 16 ? gkb : 16;             // K blocks per fold chunk
    const int nch = gkb ? (pl.nkb + cb - 1) / cb : 0;
    if (gkb) {
        if (P > nch) P = nch;
        if ((size_t)pl.tiles * nch * M * kTileRows * 4 > kGroupPartBytes) P = 1;
    }
    if (P > pl.nkb) P = pl.nkb;
    if (P > 64) P = 64;
    // pieces of whole weight loads (kWBlocks K blocks) and whole fold chunks, none empty
    const int align = gkb ? cb : kWBlocks;
    pl.kbp = (pl.nkb + P - 1) / P;
    pl.kbp = (pl.kbp + align - 1) / align * align;
    pl.P = (pl.nkb + pl.kbp - 1) / pl.kbp;
    if (!gkb && pl.kbp > 256) return false;
    if (pl.P > 1 && pl.tiles > kTicketSlots) return false;
    if ((int64_t)pl.tiles * pl.P > 0x7FFFFFFF) return false;
    pl.grid = pl.tiles * pl.P;
    pl.force_p = force_p;
    pl.smem = kMmaSmem;
    pl.sms = num_sms;
    pl.stages = kWStages;
    pl.stage_bytes = kWTileBytes;
    // workspace: tickets, scales (64 floats), bf16 code tiles [nkb][BN][64], then
    // int32 [P][M][128] piece sums per tile for split plans.  The region is
    // sized for any N' <= N on this device (grouped launches run one plan
    // per weight matrix): K is split when the exactness limit forces it
    // (every tile) or when a matrix has fewer tiles than 4/5 of the CTA slots.
    pl.off_sa = kTicketBytes;
    pl.off_sum = pl.off_sa + 256;  // e4m3 path: code sums [M][pieces of 4096 codes]
    pl.off_codes = round_up_sz(pl.off_sum + (size_t)M * ((K + 4095) / 4096) * 4, 256);
    // (K blocks rounded up to an even count: the e4m3 tiles cover 128 codes)
    pl.off_part = round_up_sz(pl.off_codes + (size_t)((pl.nkb + 1) / 2 * 2) * pl.BN * kKBlock * 2, 256);
    const int64_t small = 2 * num_sms * 4 / 5;
    // row-wise scales: an int32 slice [M][128] per tile and K piece.  A split
    // by the tiles keeps tiles' * P' <= the CTA slots; one forced by the
    // exactness limit or the tuning has at most tiles * max(pmin, force_p).
    int64_t units = slots;
    if (pmin > 1 && units < (int64_t)pl.tiles * pmin) units = (int64_t)pl.tiles * pmin;
    if (force_p > 1 && units < (int64_t)pl.tiles * force_p) units = (int64_t)pl.tiles * force_p;
    if (pl.P > 1 && units < (int64_t)pl.tiles * pl.P) units = (int64_t)pl.tiles * pl.P;
    // group scales: the chunk sums of a split matrix (a split needs fewer
    // tiles than 4/5 of the CTA slots and at most kGroupPartBytes of sums)
    size_t part = (size_t)units * M * kTileRows * 4;
    if (gkb) {
        const size_t tb = (size_t)(pl.tiles < small ? pl.tiles : small);
        part = nch > 1 ? tb * nch * M * kTileRows * 4 : 0;
        if (part > kGroupPartBytes) part = kGroupPartBytes;
    }
    pl.off_acc = pl.off_part + round_up_sz(part, 256);
    // the atomic accumulators (row-wise plans with more than kSliceMaxP
    // pieces), apart from the slices so that a grouped call may mix both
    const size_t accb = gkb ? 0 : (size_t)units * M * kTileRows * 4;
    pl.ws_bytes = pl.off_acc + round_up_sz(accb, 256);
    *out = pl;
    return true;
}

cudaError_t launch_w4a8_mma(const MmaPlan& pl, const uint16_t* X, const int8_t* Xq, const float* sa,
                            int M, int64_t K, int G, const uint8_t* const* Wq,
                            const float* const* sw, const int64_t* Ns, float* const* Y,
                            int32_t* acc_out, int8_t* Xq_out, float* sa_out, void* ws,
                            unsigned flags, cudaStream_t stream, int gs, const float* const* sg,
                            bool e4m3) {
    const int gkb = gs > 0 ? gs / kKBlock : 0;
    if (e4m3 && gkb) return cudaErrorInvalidValue;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    float* sa_ws = reinterpret_cast<float*>(wsb + pl.off_sa);
    uint8_t* codes = wsb + pl.off_codes;
    int pre_pieces = 0;
    {
        const __half* xh = reinterpret_cast<const __half*>(X);
        int Mi = M, BNi = pl.BN;
        int64_t Kk = K;
        int32_t* sum_part = reinterpret_cast<int32_t*>(wsb + pl.off_sum);
        // the atomic split plans' accumulators: the most tiles of any matrix
        int32_t* acc = reinterpret_cast<int32_t*>(wsb + pl.off_acc);
        int64_t acc_words = 0;
        for (int g = 0; g < G && !gkb; ++g) {
            MmaPlan pg;
            if (!make_mma_plan(M, K, Ns[g], pl.sms, &pg, 0, pl.force_p)) return cudaErrorInvalidValue;
            if (pg.P > kSliceMaxP && (int64_t)pg.tiles * M * kTileRows > acc_words)
                acc_words = (int64_t)pg.tiles * M * kTileRows;
        }
        void* args[] = {&xh, &Xq, &sa, &Mi, &Kk, &BNi, &codes, &sa_ws, &Xq_out, &sa_out, &acc, &acc_words,
                        &sum_part};
        const int64_t vecs = e4m3 ? (K + 127) / 128 * 8 : (int64_t)pl.nkb * 8;  // per batch row
        const unsigned pieces = (unsigned)((vecs + kAQThreads - 1) / kAQThreads);
        pre_pieces = (int)pieces;
        const void* pre = e4m3 ? reinterpret_cast<const void*>(act_codes_e4m3_kernel)
                               : reinterpret_cast<const void*>(act_codes_kernel);
        cudaError_t e = launch_pdl(pre, dim3(pl.BN, pieces), dim3(kAQThreads), 0, stream, flags, args);
        if (e != cudaSuccess) return e;
    }
    static int attr_set[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_set[dev]) {
        const void* fns[] = {reinterpret_cast<const void*>(mma_kernel<false, false, false>),
                             reinterpret_cast<const void*>(mma_kernel<false, false, true>),
                             reinterpret_cast<const void*>(mma_kernel<false, true, false>),
                             reinterpret_cast<const void*>(mma_kernel<false, true, true>),
                             reinterpret_cast<const void*>(mma_kernel<true, false, false>)};
        for (const void* f : fns) {
            e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kMmaSmem);
            if (e != cudaSuccess) return e;
        }
        if (e != cudaSuccess) return e;
        attr_set[dev] = 1;
    }
    for (int g = 0; g < G; ++g) {
        MmaPlan pg;
        if (!make_mma_plan(M, K, Ns[g], pl.sms, &pg, gkb, pl.force_p)) return cudaErrorInvalidValue;
        MmaArgs a;
        memset(&a, 0, sizeof(a));
        if (!encode_2d(&a.tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wq[g], (uint64_t)(K / 2), (uint64_t)Ns[g],
                       (uint64_t)(K / 2), kWBlocks * kKBlock / 2, kTileRows, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        a.codes = codes;
        a.sw = sw ? sw[g] : nullptr;
        if (gkb) {
            a.sg = sg[g];
            a.gld = (int)((K / gs + 3) / 4 * 4);
            a.gkb = gkb;
            a.part_f = reinterpret_cast<float*>(wsb + pg.off_part);
            a.nch = (pg.nkb + (gkb > 16 ? gkb : 16) - 1) / (gkb > 16 ? gkb : 16);
        }
        a.sa = sa_ws;
        a.Y = Y[g];
        a.acc_out = (G == 1) ? acc_out : nullptr;
        a.part = reinterpret_cast<int32_t*>(wsb + pg.off_part);
        a.acc = reinterpret_cast<int32_t*>(wsb + pg.off_acc);
        a.tickets = reinterpret_cast<unsigned*>(wsb);
        a.M = M;
        a.N = (int)Ns[g];
        a.K = (int)K;
        a.BN = pg.BN;
        a.P = pg.P;
        a.nkb = pg.nkb;
        a.kbp = pg.kbp;
        a.sum_part = reinterpret_cast<const int32_t*>(wsb + pl.off_sum);
        a.pre_pieces = pre_pieces;
        void* args[] = {&a};
        const bool atomic = !gkb && pg.P > kSliceMaxP;
        const void* fn = gkb ? reinterpret_cast<const void*>(mma_kernel<true, false, false>)
                       : e4m3 ? (atomic ? reinterpret_cast<const void*>(mma_kernel<false, true, true>)
                                        : reinterpret_cast<const void*>(mma_kernel<false, true, false>))
                              : (atomic ? reinterpret_cast<const void*>(mma_kernel<false, false, true>)
                                        : reinterpret_cast<const void*>(mma_kernel<false, false, false>));
        e = launch_pdl(fn, dim3(pg.grid), dim3(kMmaThreads),
                       kMmaSmem, stream, flags, args);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t read_and_clear_mma_error(unsigned* flags, cudaStream_t stream) {
    unsigned v = 0, z = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_mma_error, sizeof(v), 0, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbolAsync(g_mma_error, &z, sizeof(z), 0, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    *flags |= v;
    return e;
}

}  // namespace w4a8
