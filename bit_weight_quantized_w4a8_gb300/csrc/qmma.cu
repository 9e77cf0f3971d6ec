// qmma.cu -- W4A8 linear for decode batches of 2..32 rows on the warp-level
// MMA (mma.sync, fp32 accumulation), operands built in registers: e4m3
// (m16n8k32, the default) or binary16 (m16n8k16).
//
// The arithmetic is the W4A8 contract of the Jetson INT4 page (sections
// 正确方向 / 当前实现方式): INT8 activation codes times INT4 weight codes,
// summed exactly in integers, y = ((float)acc * s_w) * s_a.
//
// e4m3 operand encodings (all exact):
//  * weights: a packed nibble n (two's complement code q) becomes the byte
//    v = n ^ 8 = q + 8 in [0, 15].  Read as e4m3, a byte whose bits 4..6
//    are zero is exactly v * 2^-9: bytes 0..7 are the subnormals m * 2^-9
//    and bytes 8..15 the first binade (8 + m) * 2^-9.  Eight codes of a
//    packed word turn into two registers of four such bytes with one xor,
//    one shift and two masks: no lookup, no conversion instruction.
//  * activations: an INT8 code a is split as a = 16 a_hi + a_lo with
//    a_hi = a >> 4 in [-8, 7] and a_lo = a & 15 in [0, 15]; both are small
//    integers, exact in e4m3.  Batch row m takes two MMA columns (a_hi and
//    a_lo), so an n-tile of 8 columns covers 4 batch rows.
//  * products and sums: v * 2^-9 times an e4m3 integer is exact in fp32,
//    and the fp32 sums stay exact while |sum| < 2^24 * 2^-9: each warp sums
//    at most 65536 codes (|v a_lo| <= 225), which the plan guarantees.
//    Then U = 512 * D is an exact integer, and
//      acc = 16 U_hi + U_lo - 8 S_a,   S_a = sum_k a_k,
//    removes the +8 bias of the weight encoding (S_a is computed exactly
//    by the activation pass).  The result is bit-identical to the integer
//    definition, whatever the order of the hardware's sums.
// binary16 operands: the weight and activation codes themselves, exact
// binary16 integers (int4x8_to_h2 below); an n-tile covers 8 batch rows, no
// bias; |q a| <= 1016, so each warp sums at most 16384 codes.
//
// Two kernels:
//  * qmma_codes_kernel<kH> (grid: padded batch rows x pieces of 2048
//    codes): the per-row INT8 quantization (actq.cuh) or the given int8
//    codes, written in the order the MMA fragments read them (one
//    contiguous activation slice per 256-code box), and per piece the exact
//    partial sum of the row's codes.
//  * qmma_kernel<NT, R, kPersist, kH> (8 MMA warps; thread 0 fills a ring
//    of 2-D TMA boxes of 128 rows x 256 codes (128-byte swizzle) plus the
//    matching activation slices, the last warp done with a stage refills
//    it): MMA warp (wr, wk) owns R 16-row tiles and every R-th box, so the
//    activation fragments it loads serve R weight tiles; the warps' exact
//    integer sums meet in shared memory and K pieces meet in int32 through
//    the workspace (order-free).  A CTA takes one 128-row tile and K piece,
//    or (kPersist) walks tiles b, b + grid, ... through one ring.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>

#include "actq.cuh"
#include "kernels.h"
#include "plan.h"
#include "ptx.cuh"
#include "qmma_plan.h"
#include "tc.cuh"

namespace w4a8 {

__device__ unsigned g_qmma_error;  // wait timeouts of this path (same bits as the GEMV's)

namespace {

constexpr int kTile = 128;                        // weight rows per CTA
constexpr int kBoxCodes = 256;                    // K codes per box (128 bytes of a row)
constexpr int kBoxBytes = kTile * kBoxCodes / 2;  // 16384
constexpr int kMmaWarps = 8;
constexpr int kQThreads = kMmaWarps * 32;         // two warps per SM sub-partition: up to 255 registers
constexpr int kPreThreads = 256;
constexpr int kPreCodes = kPreThreads * 8;        // codes per activation-pass CTA
constexpr int kMaxNS = 8;
constexpr int kSmemMax = 227 * 1024;
constexpr int kSmemMax2 = 233472 / 2 - 1024;      // per CTA with two CTAs on an SM

struct QmmaArgs {
    CUtensorMap tmW;        // packed weights [N][K/2] uint8, box 128 bytes x 128 rows, 128B swizzle
    const uint8_t* codes;   // activation slices [nbox][8][8 NT][4][8] e4m3 bytes
    const float* sw;        // [N]
    const float* sa;        // [M]
    const int32_t* sum_part;  // [M][pre_pieces] partial sums of the activation codes
    float* Y;               // [M][N]
    int32_t* acc_out;       // optional [M][N]
    int32_t* part;          // [tiles][M][128] int32 sums when P > 1 (zeroed by the activation pass)
    unsigned* tickets;      // [tiles] when P > 1, zero between calls
    int M, N, nbox, bpp, P, NS, pre_pieces, tiles;
    unsigned long long stall_ns;  // > 0: test of the bounded waits (see qmma_kernel)
};

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
        #pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            atomicOr(&g_qmma_error, kErrFullWait);
            return false;
        }
    }
}

// Waits (bounded) until the stage's copy of CTA box j has been issued:
// tag is the box last issued into the stage.  A warp may reach box j while
// its stage still holds box j - NS (the other warps have not released it);
// the mbarrier parity alone cannot tell that phase from box j's.
__device__ __forceinline__ bool wait_issued(const volatile int* tag, int j, volatile int* abort_flag) {
    if (*tag == j) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
        #pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (*tag == j) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            atomicOr(&g_qmma_error, kErrFullWait);
            return false;
        }
    }
}

// e4m3 encoding of a small integer (|v| <= 15, exact): sign, exponent
// floor(log2 |v|) + 7, the three bits below the leading one.
__device__ __forceinline__ uint32_t e4m3_small(int v) {
    const uint32_t x = (uint32_t)(v < 0 ? -v : v);
    if (x == 0u) return 0u;
    const int e = 31 - __clz((int)x);
    return (v < 0 ? 0x80u : 0u) | ((uint32_t)(e + 7) << 3) | (((x << 3) >> e) & 7u);
}

__device__ __forceinline__ uint32_t e4m3_int4(int v0, int v1, int v2, int v3) {
    return e4m3_small(v0) | (e4m3_small(v1) << 8) | (e4m3_small(v2) << 16) | (e4m3_small(v3) << 24);
}

// Two small integers (|v| <= 2048, exact) as a binary16 pair: lo in bits 0..15.
__device__ __forceinline__ uint32_t half2_bits(int lo, int hi) {
    const __half2 h = __halves2half2(__int2half_rn(lo), __int2half_rn(hi));
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Eight packed INT4 codes (a 32-bit word, code i in bits 4i..4i+3, two's
// complement) as four binary16 pairs of the codes themselves, exactly:
// p[0] = (c0, c4), p[1] = (c1, c5), p[2] = (c2, c6), p[3] = (c3, c7).  The
// nibble n ^ 8 = q + 8 is placed under the exponent of 1024 (bits 0x6400 of
// each half): 1024 + (q + 8), minus 1032, is q; the odd codes sit 4 bits
// higher, 1024 + 16 (q + 8), and one fused multiply-add by 1/16 and -72
// gives q (every step exact in binary16).
__device__ __forceinline__ void int4x8_to_h2(uint32_t w, uint32_t p[4]) {
    const uint32_t x = w ^ 0x88888888u;
    const uint32_t y = x >> 8;
    const __half2 bias = __halves2half2(__ushort_as_half((unsigned short)0x6408u),
                                        __ushort_as_half((unsigned short)0x6408u));  // 1032
    const __half2 sc = __halves2half2(__ushort_as_half((unsigned short)0x2C00u),
                                      __ushort_as_half((unsigned short)0x2C00u));    // 1/16
    const __half2 off = __halves2half2(__ushort_as_half((unsigned short)0xD480u),
                                       __ushort_as_half((unsigned short)0xD480u));   // -72
    uint32_t u[4] = {(x & 0x000F000Fu) | 0x64006400u, (x & 0x00F000F0u) | 0x64006400u,
                     (y & 0x000F000Fu) | 0x64006400u, (y & 0x00F000F0u) | 0x64006400u};
    #pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 h = *reinterpret_cast<const __half2*>(&u[i]);
        const __half2 r = (i & 1) ? __hfma2(h, sc, off) : __hsub2(h, bias);
        p[i] = *reinterpret_cast<const uint32_t*>(&r);
    }
}

// Activation pass.  Grid (MP rows, pieces of 2048 codes covering whole
// boxes); thread u of piece y handles the 8 codes 8w..8w+7 of its row,
// w = 256 y + u.  Codes are quantized as in the other paths (or taken from
// Xq), split into a_hi / a_lo and written as e4m3 bytes where the MMA
// fragments read them: in box b, code 256 b + 32 s + 8 t + e (s in 0..7,
// t in 0..3, e in 0..7) belongs to K step s and lane column t; its even
// elements e go to fragment register b0, the odd ones to b1;
// batch row m is column 8 (m / 4) + 2 (m % 4) (a_hi) and the next one
// (a_lo).  Slice layout: [box][s][column][t][b0 (4 bytes), b1 (4 bytes)].
// Rows m >= M and codes past K are zero.  Each CTA also writes the sum of
// its piece's codes of row m (exact int32) and clears the split-K
// accumulators.
// kH (binary16 operands): the codes themselves, exact binary16 integers, in
// the order of the m16n8k16 B fragments: C = 8 NT columns are NT n-tiles of
// 8 batch rows (row m: n-tile m / 8, fragment column g = m % 8); 16-byte
// chunk cc of a box holds K sub-steps s = 0, 1, and lane (g, t) of sub-step
// s takes codes (8t + 2s, 8t + 2s + 4) as b0 and (8t + 2s + 1, 8t + 2s + 5)
// as b1 of the chunk (the pairs the weight conversion forms).  Slice
// layout: [box][cc][s][n-tile][lane][b0, b1], 512 C bytes a box.
template <bool kH>
__global__ void __launch_bounds__(kPreThreads) qmma_codes_kernel(
    const __half* __restrict__ X, const int8_t* __restrict__ Xq, const float* __restrict__ sa_in,
    int M, int64_t K, int C, int64_t words, uint8_t* __restrict__ codes, float* __restrict__ sa_ws,
    int32_t* __restrict__ sum_part, int8_t* __restrict__ Xq_out, float* __restrict__ sa_out,
    int32_t* __restrict__ acc, int64_t acc_words) {
    __shared__ float red[kPreThreads / 32];
    __shared__ int isum[kPreThreads / 32];
    griddep_launch_dependents();
    griddep_wait();
    for (int64_t e = ((int64_t)blockIdx.y * gridDim.x + blockIdx.x) * kPreThreads + threadIdx.x; e < acc_words;
         e += (int64_t)gridDim.x * gridDim.y * kPreThreads)
        acc[e] = 0;
    const int m = blockIdx.x;
    const int64_t w = (int64_t)blockIdx.y * kPreThreads + threadIdx.x;  // 8-code word of the row
    const int64_t kchunks = K / 8;
    const bool real = m < M;
    float s = 0.f;
    const uint4* xv = reinterpret_cast<const uint4*>(X + (int64_t)(real ? m : 0) * K);
    if (real) {
        if (X == nullptr) {
            s = sa_in[m];
        } else {
            __half2 hm = __float2half2_rn(0.f);
            #pragma unroll 4
            for (int64_t v = threadIdx.x; v < kchunks; v += kPreThreads) {
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
            for (int i = 0; i < kPreThreads / 32; ++i) mx = fmaxf(mx, red[i]);
            s = __fdiv_rn(mx, 127.f);
        }
    }
    int rsum = 0;
    if (w < words) {
        uint32_t ev = 0u, od = 0u;  // int8 codes of the even / odd elements
        if (real && w < kchunks) {
            if (X != nullptr) {
                float r_lo, r_hi;
                quant_bracket(s, &r_lo, &r_hi);
                const uint2 q = quant8_split(xv[w], s, r_lo, r_hi);
                ev = q.x;
                od = q.y;
                if (Xq_out != nullptr)
                    *reinterpret_cast<uint2*>(Xq_out + (int64_t)m * K + 8 * w) =
                        make_uint2(__byte_perm(q.x, q.y, 0x5140), __byte_perm(q.x, q.y, 0x7362));
            } else {
                const uint2 c = *reinterpret_cast<const uint2*>(Xq + (int64_t)m * K + 8 * w);
                ev = __byte_perm(c.x, c.y, 0x6420);
                od = __byte_perm(c.x, c.y, 0x7531);
            }
        }
        int e[4], o[4];
        #pragma unroll
        for (int i = 0; i < 4; ++i) {
            e[i] = (int)(int8_t)((ev >> (8 * i)) & 0xFFu);
            o[i] = (int)(int8_t)((od >> (8 * i)) & 0xFFu);
            rsum += e[i] + o[i];
        }
        // word w of the row: box b, K step (16-byte chunk) sidx, lane column t
        const int64_t b = w >> 5;
        const int sidx = (int)(w >> 2) & 7, t = (int)w & 3;
        if constexpr (kH) {
            // code 2i is e[i], code 2i + 1 is o[i]
            const int nt = m >> 3, g = m & 7;
            uint8_t* base = codes + b * ((int64_t)512 * C) + (int64_t)nt * 256 + (g * 4 + t) * 8;
            #pragma unroll
            for (int sub = 0; sub < 2; ++sub)
                *reinterpret_cast<uint2*>(base + (int64_t)(sidx * 2 + sub) * (C / 8) * 256) =
                    make_uint2(half2_bits(e[sub], e[sub + 2]), half2_bits(o[sub], o[sub + 2]));
        } else {
            const int col = 8 * (m >> 2) + 2 * (m & 3);
            uint8_t* base = codes + b * ((int64_t)256 * C) + ((int64_t)(sidx * C + col) * 4 + t) * 8;
            const uint2 hi = make_uint2(e4m3_int4(e[0] >> 4, e[1] >> 4, e[2] >> 4, e[3] >> 4),
                                        e4m3_int4(o[0] >> 4, o[1] >> 4, o[2] >> 4, o[3] >> 4));
            const uint2 lo = make_uint2(e4m3_int4(e[0] & 15, e[1] & 15, e[2] & 15, e[3] & 15),
                                        e4m3_int4(o[0] & 15, o[1] & 15, o[2] & 15, o[3] & 15));
            *reinterpret_cast<uint2*>(base) = hi;
            *reinterpret_cast<uint2*>(base + 32) = lo;  // the next column
        }
    }
    // the piece's exact sum of codes (|sum| <= 127 * 2048)
    #pragma unroll
    for (int o = 16; o >= 1; o >>= 1) rsum += __shfl_xor_sync(0xFFFFFFFFu, rsum, o);
    if ((threadIdx.x & 31) == 0) isum[threadIdx.x >> 5] = rsum;
    __syncthreads();
    if (threadIdx.x == 0 && real) {
        int tsum = 0;
        #pragma unroll
        for (int i = 0; i < kPreThreads / 32; ++i) tsum += isum[i];
        sum_part[(int64_t)m * gridDim.y + blockIdx.y] = tsum;
        if (blockIdx.y == 0) {
            sa_ws[m] = s;
            if (sa_out != nullptr) sa_out[m] = s;
        }
    }
}

// Four 8x8 b16 matrices from shared memory: lanes 8q..8q+7 give the 16-byte
// row addresses of matrix q; lane (g, t) receives 4 bytes (t) of row g of
// each matrix.
__device__ __forceinline__ void ldmatrix_x4(uint32_t* d, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
                 : "r"(addr));
}

__device__ __forceinline__ void mma_f16(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_e4m3(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Shared memory (base aligned to 1024 for the swizzled boxes): NS stages of
// [weight box 16384][activation slice 2048 NT], the integer row sums
// [128][4 NT] int32, the activation sums [4 NT], NS mbarriers (stage
// landed), per stage the number of warps done with it and the last box
// copied into it, the abort and last-CTA flags.
//
// MMA warp w is (wr, wk) = (w % (8 / R), w / (8 / R)): weight rows
// 16 R wr .. 16 R wr + 16 R - 1 (R m16 tiles) of every box i of the piece
// with i % R == wk (R = 1: every warp takes every box, 16 rows each).
// Lane (g, t) = (lane / 4, lane % 4) of a tile holds fragment rows g and
// g + 8, which are tile rows pi(g) and pi(g) + 8 with
// pi = (0, 4, 1, 5, 2, 6, 3, 7).  K step s of a box is the 16-byte chunk s
// of every row: ldmatrix gives lane (g, t) word t of that chunk of rows
// pi(g) and pi(g) + 8 (8 codes each: the even ones are fragment columns
// 4t..4t+3, the odd ones 16+4t..16+4t+3); with the 128-byte swizzle (chunk
// c of row r at r * 128 + (c ^ (r % 8)) * 16) the eight rows of each
// matrix sit in eight different bank groups.  KS accumulator sets take
// alternate K steps, so that a warp with few tiles still has 2 R NT
// independent MMA chains.  There is no copy warp: thread 0 fills the
// ring at entry, and the last warp done with a stage refills it with the
// box NS further on.
//
// kPersist (one K piece, more tiles than SMs): CTA b takes the tiles
// b, b + grid, ... and streams their boxes as one sequence j = ti * nb + i
// (local tile ti, box i) through the ring, so the copies of the next tile
// are in flight while a tile ends; after a tile's last box the warps' sums
// meet in shared memory, the CTA writes the tile's outputs and clears the
// sums.  Without it a CTA takes one tile and K piece (grid tiles x P).
// Persistent CTAs of up to 8 batch rows (at most 2 n-tiles) run two to an
// SM: their latency-bound warps then have twice the company (128 registers
// a thread, which those instantiations fit without spilling).
//
// kH (binary16 operands, mma.sync m16n8k16 f16 -> f32): a weight word
// becomes four pairs of the codes themselves (int4x8_to_h2), the
// activation codes are exact binary16 integers, an n-tile covers 8 batch
// rows (no high / low split) and no bias is removed.  Products |q a| <=
// 1016 and every fp32 sum of one warp's boxes (at most 16384 codes, which
// the plan guarantees) stay below 2^24: exact.  Of a 16-byte chunk, K
// sub-step s pairs (c 2s, c 2s + 4) of word t as fragment columns 2t, 2t + 1
// and (c 2s + 1, c 2s + 5) as 2t + 8, 2t + 9.
template <int NT, int R, bool kPersist, bool kH>
__global__ void __launch_bounds__(kQThreads, (kPersist && NT <= 2) ? 2 : 1)
    qmma_kernel(const __grid_constant__ QmmaArgs a) {
    constexpr int C = 8 * NT;        // MMA columns
    constexpr int MP = (kH ? 8 : 4) * NT;  // batch rows covered
    constexpr int kActBytes = (kH ? 512 : 256) * C;
    constexpr int kStage = kBoxBytes + kActBytes;
    constexpr int WR = kMmaWarps / R;  // warps per box
    constexpr int KS = R * NT <= 2 ? 2 : 1;  // accumulator sets (alternate K steps)
    constexpr bool kUnroll = R * NT <= 4;    // the four K-step pairs of a box unrolled
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const int NS = a.NS;
    int* red = reinterpret_cast<int*>(smem + NS * kStage);
    int* sa_sum = red + kTile * MP;
    uint64_t* full = reinterpret_cast<uint64_t*>(sa_sum + MP);
    int* released = reinterpret_cast<int*>(full + NS);
    int* last_box = released + NS;
    volatile int* abort_flag = last_box + NS;
    int* last_flag = last_box + NS + 1;
    uint64_t* never = reinterpret_cast<uint64_t*>(last_box + NS + 2);  // 8-byte aligned (16 NS + 8 past full)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = kPersist ? (int)blockIdx.x : (int)blockIdx.x / a.P;  // (first) tile
    const int p = kPersist ? 0 : (int)blockIdx.x % a.P;
    const int box0 = p * a.bpp;
    const int nb = min(a.bpp, a.nbox - box0);
    const int ntl = kPersist ? (a.tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 1;
    const int total = ntl * nb;  // boxes this CTA streams
    const uint64_t pol_w = l2_evict_first_policy();
    const uint64_t pol_a = l2_evict_last_policy();
    // CTA box j = ti * nb + i: box box0 + i of local tile ti, into stage j % NS
    auto issue_w = [&](int j) {
        const int ti = kPersist ? j / nb : 0;
        const int i = j - ti * nb;
        tma_load_2d_hint(smem_u32(smem + (j % NS) * kStage), &a.tmW, (box0 + i) * (kBoxCodes / 2),
                         (tile + ti * (int)gridDim.x) * kTile, smem_u32(full + j % NS), pol_w);
    };
    auto issue_a = [&](int j) {
        const int i = kPersist ? j % nb : j;
        bulk_g2s(smem_u32(smem + (j % NS) * kStage + kBoxBytes), a.codes + (int64_t)(box0 + i) * kActBytes,
                 kActBytes, smem_u32(full + j % NS), pol_a);
    };

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_u32(full + s), 1);
            released[s] = 0;
            last_box[s] = -1;
        }
        mbar_init(smem_u32(never), 1);  // nothing ever arrives on it
        *abort_flag = 0;
        fence_mbar_init();
    }
    for (int e = tid; e < kTile * MP + MP; e += kQThreads) red[e] = 0;  // row sums, activation sums
    __syncthreads();
    griddep_launch_dependents();
    const int pre = min(NS, total);
    if (tid == 0) {  // the weights do not depend on earlier launches
        for (int j = 0; j < pre; ++j) {
            mbar_arrive_expect_tx(smem_u32(full + j), kStage);
            issue_w(j);
            last_box[j] = j;
        }
    }
    griddep_wait();  // activation slices, sums, scales, outputs and workspace from here on
    if (tid == 0)
        for (int j = 0; j < pre; ++j) issue_a(j);
    // the batch rows' exact code sums, from the activation pass's pieces
    // (one load per thread, added in shared memory; read after the loop)
    if constexpr (!kH)  // binary16 codes carry no bias: the sums stay 0
        for (int e = tid; e < a.M * a.pre_pieces; e += kQThreads)
            atomicAdd(sa_sum + e / a.pre_pieces, __ldcg(a.sum_part + e));

    const int wr = warp % WR, wk = warp / WR;
    const int g = lane >> 2, t = lane & 3;
    const int pg = (g >> 1) + 4 * (g & 1);
    // ldmatrix row of this lane: lanes 8 q .. 8 q + 7 address matrix q = (rows
    // g or g + 8) x (chunk 2 sp or 2 sp + 1) of tile rt; row pi(lane % 8)
    const int lg = lane & 7;
    const int lsw = (lg >> 1) + 4 * (lg & 1);
    const uint32_t lrow = (uint32_t)((16 * R * wr + lsw + 8 * ((lane >> 3) & 1)) * 128);
    const int lchunk = lane >> 4;
    if (a.stall_ns != 0ull) {
        // test of the bounded waits: a wait for a phase that never completes
        // runs out after stall_ns, sets the error word and the abort flag;
        // the loop below then stops at the first stage not yet landed, and
        // the copies in flight are waited for before the CTA exits
        __all_sync(0xFFFFFFFFu, wait_bounded(smem_u32(never), 0, abort_flag, a.stall_ns));
    }
    #pragma unroll 1
    for (int ti = 0; ti < ntl; ++ti) {
    float acc[KS][R][NT][4];
    #pragma unroll
    for (int k = 0; k < KS; ++k)
        #pragma unroll
        for (int rt = 0; rt < R; ++rt)
            #pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                #pragma unroll
                for (int i = 0; i < 4; ++i) acc[k][rt][nt][i] = 0.f;
    #pragma unroll 1
    for (int i = wk; i < nb; i += R) {
        const int j = ti * nb + i;  // CTA box
        const int s = j % NS;
        if (!__all_sync(0xFFFFFFFFu, wait_issued(last_box + s, j, abort_flag))) break;
        if (!__all_sync(0xFFFFFFFFu, wait_bounded(smem_u32(full + s), (uint32_t)(j / NS) & 1u, abort_flag, kWaitLimitNs)))
            break;
        const uint32_t wbox = smem_u32(smem + s * kStage) + lrow;
        const uint8_t* abox = smem + s * kStage + kBoxBytes + (g * 4 + t) * 8;
        #pragma unroll (kUnroll ? 4 : 1)
        for (int sp = 0; sp < 4; ++sp) {  // pairs of K steps (16-byte chunks 2 sp, 2 sp + 1)
            uint32_t wv[R][4];
            #pragma unroll
            for (int rt = 0; rt < R; ++rt)
                ldmatrix_x4(wv[rt], wbox + rt * 2048 + (((2 * sp + lchunk) ^ lsw) << 4));
            if constexpr (kH) {
                #pragma unroll
                for (int h = 0; h < 2; ++h) {  // chunk cc = 2 sp + h of rows g (word 2h) and g + 8 (2h + 1)
                    const int cc = 2 * sp + h;
                    uint32_t pg_[R][4], p8_[R][4];
                    #pragma unroll
                    for (int rt = 0; rt < R; ++rt) {
                        int4x8_to_h2(wv[rt][2 * h], pg_[rt]);
                        int4x8_to_h2(wv[rt][2 * h + 1], p8_[rt]);
                    }
                    #pragma unroll
                    for (int sub = 0; sub < 2; ++sub) {
                        uint2 b[NT];
                        #pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            b[nt] = *reinterpret_cast<const uint2*>(abox + ((cc * 2 + sub) * NT + nt) * 256);
                        #pragma unroll
                        for (int rt = 0; rt < R; ++rt)
                            #pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
                                mma_f16(acc[KS == 2 ? sub : 0][rt][nt], pg_[rt][2 * sub], p8_[rt][2 * sub],
                                        pg_[rt][2 * sub + 1], p8_[rt][2 * sub + 1], b[nt].x, b[nt].y);
                    }
                }
            } else {
                #pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int ks = 2 * sp + h;
                    uint2 b[NT];
                    #pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        b[nt] = *reinterpret_cast<const uint2*>(abox + (ks * C + 8 * nt) * 32);
                    #pragma unroll
                    for (int rt = 0; rt < R; ++rt) {
                        const uint32_t x0 = wv[rt][2 * h] ^ 0x88888888u, x1 = wv[rt][2 * h + 1] ^ 0x88888888u;
                        const uint32_t a0 = x0 & 0x0F0F0F0Fu, a2 = (x0 >> 4) & 0x0F0F0F0Fu;
                        const uint32_t a1 = x1 & 0x0F0F0F0Fu, a3 = (x1 >> 4) & 0x0F0F0F0Fu;
                        #pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            mma_e4m3(acc[KS == 2 ? h : 0][rt][nt], a0, a1, a2, a3, b[nt].x, b[nt].y);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) {
            // the last warp done with this stage refills it with the box NS further on
            __threadfence_block();
            if (atomicAdd(released + s, 1) == WR - 1) {
                released[s] = 0;
                __threadfence_block();
                if (j + NS < total && !*abort_flag) {
                    mbar_arrive_expect_tx(smem_u32(full + s), kStage);
                    issue_w(j + NS);
                    issue_a(j + NS);
                    __threadfence_block();
                    last_box[s] = j + NS;
                }
            }
        }
    }
    // exact integers: U = 512 D, row value 16 U_hi + U_lo (batch row 4 nt + t);
    // binary16: D itself, columns 2t and 2t + 1 of n-tile nt are batch rows
    // 8 nt + 2t and 8 nt + 2t + 1
    #pragma unroll
    for (int rt = 0; rt < R; ++rt) {
        const int r0 = 16 * (R * wr + rt) + pg;
        if constexpr (kH) {
            #pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int m = 8 * nt + 2 * t;
                int v[4] = {0, 0, 0, 0};
                #pragma unroll
                for (int k = 0; k < KS; ++k)
                    #pragma unroll
                    for (int i = 0; i < 4; ++i) v[i] += __float2int_rn(acc[k][rt][nt][i]);
                atomicAdd(red + r0 * MP + m, v[0]);
                atomicAdd(red + r0 * MP + m + 1, v[1]);
                atomicAdd(red + (r0 + 8) * MP + m, v[2]);
                atomicAdd(red + (r0 + 8) * MP + m + 1, v[3]);
            }
        } else {
            #pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int m = 4 * nt + t;
                int v0 = 0, v1 = 0;
                #pragma unroll
                for (int k = 0; k < KS; ++k) {
                    v0 += 16 * __float2int_rn(acc[k][rt][nt][0] * 512.f) + __float2int_rn(acc[k][rt][nt][1] * 512.f);
                    v1 += 16 * __float2int_rn(acc[k][rt][nt][2] * 512.f) + __float2int_rn(acc[k][rt][nt][3] * 512.f);
                }
                atomicAdd(red + r0 * MP + m, v0);
                atomicAdd(red + (r0 + 8) * MP + m, v1);
            }
        }
    }
    __syncthreads();
    if constexpr (kPersist) {
        // the abort flag is read by every thread between the two barriers,
        // where no thread can set it: the break is CTA-uniform
        if (*abort_flag) break;
        const int n0 = (tile + ti * (int)gridDim.x) * kTile;
        for (int e = tid; e < a.M * kTile; e += kQThreads) {
            const int m = e / kTile, r = e % kTile, n = n0 + r;
            const int32_t v = red[r * MP + m] - 8 * sa_sum[m];
            red[r * MP + m] = 0;  // each sum is read and cleared by one thread; rows m >= M stay 0
            if (n >= a.N) continue;
            const int64_t o = (int64_t)m * a.N + n;
            a.Y[o] = __fmul_rn(__fmul_rn(__int2float_rn(v), a.sw[n]), a.sa[m]);
            if (a.acc_out != nullptr) a.acc_out[o] = v;
        }
        __syncthreads();
    }
    }  // tiles
    if (*abort_flag && tid == 0) {
        // copies may still be landing after an abandoned wait: wait for the
        // last one of each stage (bounded) so none writes shared memory after exit
        for (int s = 0; s < NS; ++s)
            if (last_box[s] >= 0 && !mbar_wait(smem_u32(full + s), (uint32_t)(last_box[s] / NS) & 1u))
                atomicOr(&g_qmma_error, kErrDrainWait);
    }
    if constexpr (kPersist) return;
    const bool ok = *abort_flag == 0;
    const int n0 = tile * kTile;
    if (a.P == 1) {
        if (!ok) return;
        for (int e = tid; e < a.M * kTile; e += kQThreads) {
            const int m = e / kTile, r = e % kTile, n = n0 + r;
            if (n >= a.N) continue;
            const int32_t v = red[r * MP + m] - 8 * sa_sum[m];
            const int64_t o = (int64_t)m * a.N + n;
            a.Y[o] = __fmul_rn(__fmul_rn(__int2float_rn(v), a.sw[n]), a.sa[m]);
            if (a.acc_out != nullptr) a.acc_out[o] = v;
        }
        return;
    }
    // ------------------------------------------------ split K: last CTA rescales
    int32_t* acc_t = a.part + (int64_t)tile * a.M * kTile;
    if (ok)
        for (int e = tid; e < a.M * kTile; e += kQThreads) {
            const int m = e / kTile, r = e % kTile;
            atomicAdd(acc_t + e, red[r * MP + m]);  // exact, order-free
        }
    __threadfence();
    __syncthreads();
    if (tid == 0) *last_flag = (atomicAdd(a.tickets + tile, 1u) == (unsigned)(a.P - 1));
    __syncthreads();
    if (!*last_flag) return;
    __threadfence();
    for (int e = tid; e < a.M * kTile; e += kQThreads) {
        const int m = e / kTile, r = e % kTile, n = n0 + r;
        const int32_t tot = __ldcg(acc_t + e);
        __stcg(acc_t + e, 0);  // clear for the next matrix of a grouped call
        if (n >= a.N) continue;
        const int32_t v = tot - 8 * sa_sum[m];
        const int64_t o = (int64_t)m * a.N + n;
        a.Y[o] = __fmul_rn(__fmul_rn(__int2float_rn(v), a.sw[n]), a.sa[m]);
        if (a.acc_out != nullptr) a.acc_out[o] = v;
    }
    if (tid == 0) a.tickets[tile] = 0u;  // ready for the next call
}

// --------------------------------------------------------------- host side

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

// Default 16-row tiles per warp for NT n-tiles.  R = 1: all eight warps
// read every box; larger R lets one activation fragment serve R weight tiles
// (shared-memory reads of activations are NT / R times those of weights)
// and gives each warp R times the independent MMA chains, with R boxes in
// use at a time.  Measured on GB300 (gate 3584 -> 18944, 2 / 4 / 8 rows):
// R = 1: 14.3 / 15.0 / 17.9 us, R = 2: 11.7 / 12.4 / 15.2, R = 4: 11.0 /
// 11.5 / 14.6; past 4 n-tiles 4 tiles a warp would spill.
constexpr int default_r(int NT) { return NT <= 4 ? 4 : 2; }

template <int NT, int R, bool kH>
const void* kernel_ntr(bool persist) {
    // the persistent form exists for the default tiles per warp only
    if (persist) {
        if constexpr (R == default_r(NT)) return reinterpret_cast<const void*>(qmma_kernel<NT, R, true, kH>);
        return nullptr;
    }
    return reinterpret_cast<const void*>(qmma_kernel<NT, R, false, kH>);
}

template <int NT, bool kH>
const void* kernel_nt(int R, bool persist) {
    if (R == 1) return kernel_ntr<NT, 1, kH>(persist);
    if (R == 2) return kernel_ntr<NT, 2, kH>(persist);
    if constexpr (NT <= 4) {  // 4 tiles a warp would spill past 4 n-tiles
        if (R == 4) return kernel_ntr<NT, 4, kH>(persist);
    }
    return nullptr;
}

// NT: n-tiles of 4 batch rows (e4m3) or of 8 (binary16, at most 4)
const void* kernel_for(int NT, int R, bool persist, bool h16) {
    if (h16) {
        switch (NT) {
            case 1: return kernel_nt<1, true>(R, persist);
            case 2: return kernel_nt<2, true>(R, persist);
            case 3: return kernel_nt<3, true>(R, persist);
            case 4: return kernel_nt<4, true>(R, persist);
            default: return nullptr;
        }
    }
    switch (NT) {
        case 1: return kernel_nt<1, false>(R, persist);
        case 2: return kernel_nt<2, false>(R, persist);
        case 3: return kernel_nt<3, false>(R, persist);
        case 4: return kernel_nt<4, false>(R, persist);
        case 5: return kernel_nt<5, false>(R, persist);
        case 6: return kernel_nt<6, false>(R, persist);
        case 7: return kernel_nt<7, false>(R, persist);
        case 8: return kernel_nt<8, false>(R, persist);
        default: return nullptr;
    }
}

cudaError_t set_attributes() {
    static bool done[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && done[dev]) return cudaSuccess;
    for (int nt = 1; nt <= kQmmaMaxM / 4; ++nt)
        for (int r = 1; r <= 4; r *= 2)
            for (int v = 0; v < 4; ++v) {  // persist x binary16
                const void* fn = kernel_for(nt, r, (v & 1) != 0, (v & 2) != 0);
                if (fn == nullptr) continue;
                e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
                if (e != cudaSuccess) return e;
            }
    if (dev < 64) done[dev] = true;
    return cudaSuccess;
}

// activation slice of one box, batch rows an n-tile covers
constexpr int act_box_bytes(int NT, bool h16) { return (h16 ? 4096 : 2048) * NT; }
constexpr int rows_per_tile(bool h16) { return h16 ? 8 : 4; }

size_t smem_bytes(int NT, int NS, bool h16) {
    const int MP = rows_per_tile(h16) * NT;
    return 1024 + (size_t)NS * (kBoxBytes + act_box_bytes(NT, h16)) + (size_t)kTile * MP * 4 + (size_t)MP * 4 +
           (size_t)NS * 8 + (size_t)(2 * NS + 2) * 4 + 16;
}

}  // namespace

// Plan: one CTA per SM for each 128-row tile and K piece.  K is split into
// pieces of whole boxes when the tiles leave more than a fifth of the SMs
// idle, and so that each MMA warp sums at most ceil(bpp / R) <= 256 boxes
// (65536 codes), which keeps its fp32 sums exact.  The ring takes up to
// kMaxNS stages of the shared memory.  R = 0 takes the default tiles per
// warp.  With one K piece, more tiles than SMs and the default R,
// persistent CTAs walk the tiles (no waves of CTAs, each paying the ring's
// fill): two per SM up to 8 rows (shared memory for both), else one.
bool make_qmma_plan(int M, int64_t K, int64_t N, int num_sms, QmmaPlan* out, int R, bool h16) {
    if (M < 2 || M > kQmmaMaxM || K < 32 || K % 32 || K > 131072 || N < 1 || N > 0x7FFFFFFF ||
        num_sms < 1)
        return false;
    QmmaPlan pl = {};
    pl.M = M;
    pl.h16 = h16 ? 1 : 0;
    pl.NT = (M + rows_per_tile(h16) - 1) / rows_per_tile(h16);
    pl.R = R == 0 ? default_r(pl.NT) : R;
    if (pl.R != 1 && pl.R != 2 && pl.R != 4) return false;
    if (pl.R == 4 && pl.NT > 4) return false;
    pl.tiles = (int)((N + kTile - 1) / kTile);
    pl.nbox = (int)((K + kBoxCodes - 1) / kBoxCodes);
    int P = 1;
    if (pl.tiles < num_sms * 4 / 5) P = num_sms / pl.tiles;
    // each warp sums at most 256 boxes (65536 codes) of e4m3 products
    // (|v a_lo| <= 225) or 64 boxes (16384 codes) of binary16 ones (|q a| <=
    // 1016): exact fp32 sums
    const int wmax = h16 ? 64 : 256;
    const int pmin = (pl.nbox + wmax * pl.R - 1) / (wmax * pl.R);
    if (P < pmin) P = pmin;
    if (P > pl.nbox) P = pl.nbox;
    if (P < 1) P = 1;
    pl.bpp = (pl.nbox + P - 1) / P;
    pl.P = (pl.nbox + pl.bpp - 1) / pl.bpp;
    if ((pl.bpp + pl.R - 1) / pl.R > wmax) return false;
    if (pl.P > 1 && pl.tiles > kTicketSlots) return false;
    if ((int64_t)pl.tiles * pl.P > 0x7FFFFFFF) return false;
    pl.persist = (pl.P == 1 && pl.tiles > num_sms && pl.R == default_r(pl.NT)) ? 1 : 0;
    const bool two = pl.persist && pl.NT <= 2;  // two persistent CTAs per SM
    const size_t cap = two ? (size_t)kSmemMax2 : (size_t)kSmemMax;
    int NS = kMaxNS < pl.bpp ? kMaxNS : pl.bpp;
    while (NS > 2 && smem_bytes(pl.NT, NS, h16) > cap) --NS;
    if (smem_bytes(pl.NT, NS, h16) > cap) return false;
    pl.NS = NS;
    pl.stage_bytes = kBoxBytes + act_box_bytes(pl.NT, h16);
    pl.smem = (int)smem_bytes(pl.NT, NS, h16);
    pl.grid = !pl.persist ? pl.tiles * pl.P : two ? (pl.tiles < 2 * num_sms ? pl.tiles : 2 * num_sms) : num_sms;
    pl.sms = num_sms;
    pl.pre_pieces = (int)(((int64_t)pl.nbox * kBoxCodes + kPreCodes - 1) / kPreCodes);
    // workspace: tickets, scales (64 floats), activation sums [M][pre_pieces],
    // activation slices [nbox][act_box_bytes], then int32 [M][128] accumulators per
    // tile for split plans.  Sized for any N' <= N on this device (grouped
    // launches plan each matrix on its own): a matrix is split only when its
    // tiles are fewer than 4/5 of the SMs or when K is longer than the
    // warps' exact range (then for every tile).
    pl.off_sa = kTicketBytes;
    pl.off_sum = pl.off_sa + 256;
    pl.off_codes = round_up_sz(pl.off_sum + (size_t)M * pl.pre_pieces * 4, 256);
    pl.off_part = round_up_sz(pl.off_codes + (size_t)pl.nbox * act_box_bytes(pl.NT, h16), 256);
    const int64_t small = num_sms * 4 / 5;
    const int64_t tmax = pmin > 1 ? pl.tiles : (pl.tiles < small ? pl.tiles : small);
    pl.ws_bytes = pl.off_part + round_up_sz((size_t)tmax * M * kTile * 4, 256);
    *out = pl;
    return true;
}

cudaError_t launch_w4a8_qmma(const QmmaPlan& pl, const uint16_t* X, const int8_t* Xq, const float* sa,
                             int M, int64_t K, int G, const uint8_t* const* Wq,
                             const float* const* sw, const int64_t* Ns, float* const* Y,
                             int32_t* acc_out, int8_t* Xq_out, float* sa_out, void* ws,
                             unsigned flags, cudaStream_t stream, unsigned long long stall_ns) {
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    float* sa_ws = reinterpret_cast<float*>(wsb + pl.off_sa);
    int32_t* sum_part = reinterpret_cast<int32_t*>(wsb + pl.off_sum);
    uint8_t* codes = wsb + pl.off_codes;
    {
        const __half* xh = reinterpret_cast<const __half*>(X);
        int Mi = M, Ci = 8 * pl.NT;
        int64_t Kk = K, words = (int64_t)pl.nbox * (kBoxCodes / 8);
        int32_t* acc = reinterpret_cast<int32_t*>(wsb + pl.off_part);
        int64_t acc_words = (int64_t)((pl.ws_bytes - pl.off_part) / 4);
        void* args[] = {&xh, &Xq, &sa, &Mi, &Kk, &Ci, &words, &codes, &sa_ws, &sum_part, &Xq_out, &sa_out,
                        &acc, &acc_words};
        const void* pre = pl.h16 ? reinterpret_cast<const void*>(qmma_codes_kernel<true>)
                                 : reinterpret_cast<const void*>(qmma_codes_kernel<false>);
        cudaError_t e = launch_pdl(pre, dim3(rows_per_tile(pl.h16 != 0) * pl.NT, pl.pre_pieces), dim3(kPreThreads), 0,
                                   stream, flags, args);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = set_attributes();
    if (e != cudaSuccess) return e;
    for (int g = 0; g < G; ++g) {
        QmmaPlan pg;
        if (!make_qmma_plan(M, K, Ns[g], pl.sms, &pg, pl.R, pl.h16 != 0)) return cudaErrorInvalidValue;
        QmmaArgs a;
        memset(&a, 0, sizeof(a));
        if (!make_w4_tile_map(&a.tmW, Wq[g], K, Ns[g])) return cudaErrorInvalidValue;
        a.codes = codes;
        a.sw = sw[g];
        a.sa = sa_ws;
        a.sum_part = sum_part;
        a.Y = Y[g];
        a.acc_out = (G == 1) ? acc_out : nullptr;
        a.part = reinterpret_cast<int32_t*>(wsb + pg.off_part);
        a.tickets = reinterpret_cast<unsigned*>(wsb);
        a.M = M;
        a.N = (int)Ns[g];
        a.nbox = pg.nbox;
        a.bpp = pg.bpp;
        a.P = pg.P;
        a.NS = pg.NS;
        a.pre_pieces = pg.pre_pieces;
        a.tiles = pg.tiles;
        a.stall_ns = stall_ns;
        const void* fn = kernel_for(pg.NT, pg.R, pg.persist != 0, pg.h16 != 0);
        if (fn == nullptr) return cudaErrorInvalidValue;
        void* args[] = {&a};
        e = launch_pdl(fn, dim3(pg.grid), dim3(kQThreads), pg.smem, stream, flags, args);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t read_and_clear_qmma_error(unsigned* flags, cudaStream_t stream) {
    unsigned v = 0, z = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_qmma_error, sizeof(v), 0, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbolAsync(g_qmma_error, &z, sizeof(z), 0, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    *flags |= v;
    return e;
}

}  // namespace w4a8
