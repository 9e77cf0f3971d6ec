// rowdot.cu -- W4A8 linear for small decode batches (2..8 activation rows)
// on the integer pipe, one weight row per thread group.
//
// The arithmetic is the W4A8 contract of the Jetson INT4 page (sections
// 正确方向 / 当前实现方式): INT8 activation codes times INT4 weight codes,
// summed exactly in int32, y = ((float)acc * s_w) * s_a.
//
// Where the dp4a GEMV spreads one weight row over a warp (each lane its own
// K slice, its own activation values), this kernel gives each weight row to
// TPR threads of one warp and walks the whole K piece with them: every
// thread of the CTA then reads the same activation words at the same time
// (shared-memory broadcasts), so the activations cost one load per batch
// row per 16 bytes for the whole warp, and the weight codes are unpacked
// once for all batch rows.  Per packed word w (8 INT4 codes, two's
// complement nibbles, low nibble first):
//   lo = (w << 4) & 0xF0F0F0F0   -> bytes 16 * q of the even codes
//   hi =  w       & 0xF0F0F0F0   -> bytes 16 * q of the odd codes
// both signed bytes, so two signed dp4a against the even and odd
// activation codes add 16 * (the 8 products) to the accumulator with no
// correction term; the sum is a multiple of 16 and >> 4 recovers it.
// |16 q a| <= 16256, so a thread's sum over at most 131072 codes stays
// inside int32.
//
// Two kernels:
//  * rowdot_codes_kernel (grid: batch rows x pieces of 2048 codes): the
//    per-row INT8 quantization of the activations (max|x|, s_a = max/127 by
//    IEEE division, round half away, clamp; actq.cuh), or the given int8
//    codes, written split by parity: per 8 codes one 8-byte word pair (the
//    4 even codes, the 4 odd codes), zero past K up to a whole 256-code box,
//    and interleaved over the batch: the 32 codes of one 16-byte weight
//    chunk are 32 contiguous bytes per batch row, the M rows of a chunk
//    adjacent ([box][chunk][M][32 bytes]).
//  * rowdot_kernel<MT, TPR> (one CTA per 128 weight rows and K piece):
//    thread 0 streams 2-D TMA boxes of 128 rows x 128 bytes (256 codes,
//    128-byte swizzle) into a ring and copies the piece's activation planes
//    once; each thread group accumulates its row's dot products with all
//    MT batch rows; pieces are summed in int32 by the CTA that finishes a
//    tile last (exact, so the result is bit-identical to the integer
//    definition whatever the split).
//  * rowdot_group_kernel<MT> (group-wise scales, 1..8 batch rows): one
//    thread per weight row, so that each row's per-group sums are folded by
//    one thread in the fixed order of the group-scale contract (below).
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
#include "tc.cuh"

namespace w4a8 {

__device__ unsigned g_rowdot_error;  // wait timeouts of this path (same bits as the GEMV's)

namespace {

constexpr int kTile = 128;             // weight rows per CTA
constexpr int kBoxCodes = 256;         // K codes per TMA box (128 bytes of a row)
constexpr int kBoxBytes = kTile * kBoxCodes / 2;  // 16384
constexpr int kActBoxBytes = kBoxCodes;           // activation bytes of one batch row per box
constexpr int kPreThreads = 256;
constexpr int kMaxNS = 8;
constexpr int kActMax = 48 * 1024;     // shared bytes for a piece's activation codes
constexpr int kSmemPerSM = 227 * 1024;

struct RowdotArgs {
    CUtensorMap tmW;        // packed weights [N][K/2] uint8, box 128 bytes x 128 rows, 128B swizzle
    const uint2* codes;     // activation codes [nbox][8][M][4] (even, odd) word pairs
    const float* sw;        // [N]
    const float* sa;        // [M]
    float* Y;               // [M][N]
    int32_t* acc_out;       // optional [M][N]
    int32_t* part;          // [tiles][P][M][128] piece sums when P > 1 (int32)
    unsigned* tickets;      // [tiles] when P > 1, zero between calls
    int M, N, nbox, bpp, P, NS;
};

// Group-wise scales: up to kGroupMats weight matrices reading the same
// activation in one launch; their 128-row tiles are numbered consecutively
// (matrix g owns tiles tile0[g] .. tile0[g + 1] - 1).
constexpr int kGroupMats = 4;
constexpr int kMaxPhases = 4;
struct GroupArgs {
    CUtensorMap tmW[kGroupMats];  // packed weights [N_g][K/2], box 128 bytes x 128 rows, 128B swizzle
    const float* sg[kGroupMats];  // [N_g][gld] fp32, one scale per 2^gshift codes
    float* Y[kGroupMats];         // [M][N_g]
    int N[kGroupMats];
    int tile0[kGroupMats + 1];    // unused matrices: tile0[g] = tile0[G]
    const uint8_t* codes;         // activation codes [nbox][8][M][32 bytes]
    const float* sa;              // [M]
    float* part_f;                // [tiles][nch][M][128] chunk sums when P > 1
    unsigned* tickets;            // [tiles] when P > 1, zero between calls
    int gshift, gld, ngroups;     // ngroups = K >> gshift
    int lshift, nch, abox;        // chunks of 2^lshift = max(group, 1024) codes, abox boxes each
    int K, M, nbox, bpp, P, NS;
    int nph;                      // thread phases (128 threads each), 1, 2 or 4
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
            atomicOr(&g_rowdot_error, kErrFullWait);
            return false;
        }
    }
}

// Waits (bounded) until ring slot `slot` holds the fill of box i: the
// thread phases of the group-scale kernel consume boxes out of order, and a
// barrier's parity alone cannot tell fill i from the fill two before it.
// last_box[slot] is the box whose fill was last issued into the slot.
__device__ __forceinline__ bool wait_slot_box(volatile int* last_box, int i, volatile int* abort_flag) {
    if (*last_box == i) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
        #pragma unroll 1
        for (int k = 0; k < 32; ++k)
            if (*last_box == i) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            atomicOr(&g_rowdot_error, kErrFullWait);
            return false;
        }
    }
}

// Activation codes.  Grid (M rows, ceil(kw / 256)); thread u handles the
// 8 codes 8u..8u+7 of row m.  Every CTA of a row takes the row's max|x|
// (exact in binary16) and s_a = max/127 by IEEE division, then quantizes its
// vectors with the fast exact quantizer; with X null it splits the given
// int8 codes Xq instead.  Optional int8 codes and scale outputs.
__global__ void __launch_bounds__(kPreThreads) rowdot_codes_kernel(
    const __half* __restrict__ X, const int8_t* __restrict__ Xq, const float* __restrict__ sa_in,
    int M, int64_t K, int64_t kw, uint2* __restrict__ codes, float* __restrict__ sa_ws,
    int8_t* __restrict__ Xq_out, float* __restrict__ sa_out) {
    __shared__ float red[kPreThreads / 32];
    griddep_launch_dependents();
    griddep_wait();
    const int m = blockIdx.x;
    const int64_t u = (int64_t)blockIdx.y * kPreThreads + threadIdx.x;
    const int64_t kchunks = K / 8;
    float s;
    const uint4* xv = reinterpret_cast<const uint4*>(X + (int64_t)m * K);
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
        for (int w = 0; w < kPreThreads / 32; ++w) mx = fmaxf(mx, red[w]);
        s = __fdiv_rn(mx, 127.f);
    }
    if (u < kw) {
        uint2 q = make_uint2(0u, 0u);
        if (u < kchunks) {
            if (X != nullptr) {
                float r_lo, r_hi;
                quant_bracket(s, &r_lo, &r_hi);
                q = quant8_split(xv[u], s, r_lo, r_hi);  // even / odd codes
                if (Xq_out != nullptr)
                    *reinterpret_cast<uint2*>(Xq_out + (int64_t)m * K + 8 * u) =
                        make_uint2(__byte_perm(q.x, q.y, 0x5140), __byte_perm(q.x, q.y, 0x7362));
            } else {
                const uint2 c = *reinterpret_cast<const uint2*>(Xq + (int64_t)m * K + 8 * u);
                q = make_uint2(__byte_perm(c.x, c.y, 0x6420), __byte_perm(c.x, c.y, 0x7531));
            }
        }
        // word pair u = (box, chunk, j): [box][chunk][m][j]
        codes[((u >> 2) * M + m) * 4 + (u & 3)] = q;
    }
    if (blockIdx.y == 0 && threadIdx.x == 0) {
        sa_ws[m] = s;
        if (sa_out != nullptr) sa_out[m] = s;
    }
}

// Shared memory (base aligned to 1024 for the swizzled boxes): the weight
// ring [NS][16384], the piece's activation codes [bpp][8][MT][32 bytes], the
// cross-warp sums [TPR - 1][MT][128] int32, NS + 1 mbarriers (ring slots,
// activations), and per slot the number of warps done with it and the last
// box copied into it.
//
// Thread mapping: warp w takes the 16-byte chunks c = w / 4 + TPR * i of
// every 128-byte box row, lane l the weight row r = (w % 4) * 32 + l.  With
// the 128-byte swizzle (chunk c of row r stored at r * 128 + ((c ^ (r % 8))
// * 16)) the eight lanes of each quarter-warp read eight different bank
// groups (conflict-free), and every activation load of a warp is one
// address (a broadcast).
template <int MT, int TPR>
__global__ void __launch_bounds__(kTile * TPR) rowdot_kernel(const __grid_constant__ RowdotArgs a) {
    constexpr int kThreads = kTile * TPR;
    constexpr int kWarps = kThreads / 32;
    constexpr int CPT = 8 / TPR;           // chunks of each box row per thread
    constexpr int kChunkAct = MT * 32;     // activation bytes of one chunk
    constexpr int kBoxAct = 8 * kChunkAct; // activation bytes of one box
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const int NS = a.NS;
    uint8_t* ring = smem;
    uint8_t* act = smem + NS * kBoxBytes;
    int* red = reinterpret_cast<int*>(act + a.bpp * kBoxAct);
    uint64_t* bars = reinterpret_cast<uint64_t*>(red + (TPR - 1) * MT * kTile);  // full[NS], activations
    int* released = reinterpret_cast<int*>(bars + NS + 1);
    int* last_box = released + NS;
    volatile int* abort_flag = last_box + NS;
    int* last_flag = last_box + NS + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x / a.P, p = blockIdx.x % a.P;
    const int box0 = p * a.bpp;
    const int nb = min(a.bpp, a.nbox - box0);
    const int t = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint64_t pol = l2_evict_first_policy();

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_u32(bars + s), 1);
            released[s] = 0;
            last_box[s] = -1;
        }
        mbar_init(smem_u32(bars + NS), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    griddep_launch_dependents();
    if (tid == 0) {  // the weights do not depend on earlier launches
        const int n0 = min(NS, nb);
        for (int i = 0; i < n0; ++i) {
            mbar_arrive_expect_tx(smem_u32(bars + i), kBoxBytes);
            tma_load_2d_hint(smem_u32(ring + i * kBoxBytes), &a.tmW, (box0 + i) * (kBoxCodes / 2),
                             tile * kTile, smem_u32(bars + i), pol);
            last_box[i] = i;
        }
    }
    griddep_wait();  // activation codes, scales, outputs and workspace from here on
    if (tid == 0) {
        const uint32_t bytes = (uint32_t)nb * kBoxAct;
        mbar_arrive_expect_tx(smem_u32(bars + NS), bytes);
        bulk_g2s(smem_u32(act), reinterpret_cast<const uint8_t*>(a.codes) + (int64_t)box0 * kBoxAct, bytes,
                 smem_u32(bars + NS), l2_evict_last_policy());
    }

    int acc[MT][2];  // 16 x the even / odd products of each batch row
    #pragma unroll
    for (int m = 0; m < MT; ++m) acc[m][0] = acc[m][1] = 0;
    const uint8_t* wrow = ring + r * 128;
    // waits end with a warp-uniform outcome (a lane may time out while
    // another sees the phase), so the warp's __syncwarp below never splits
    bool ok = __all_sync(0xFFFFFFFFu, wait_bounded(smem_u32(bars + NS), 0, abort_flag));
    int slot = 0;
    uint32_t ph = 0;
    for (int i = 0; ok && i < nb; ++i) {
        if (!__all_sync(0xFFFFFFFFu, wait_bounded(smem_u32(bars + slot), ph, abort_flag))) break;
        uint4 wv[CPT];
        #pragma unroll
        for (int ci = 0; ci < CPT; ++ci) {
            const int c = t + TPR * ci;
            wv[ci] = *reinterpret_cast<const uint4*>(wrow + slot * kBoxBytes + ((c ^ (r & 7)) << 4));
        }
        __syncwarp();
        if (lane == 0) {
            // the last warp done with this slot refills it with the box NS further on
            __threadfence_block();
            if (atomicAdd(released + slot, 1) == kWarps - 1) {
                released[slot] = 0;
                __threadfence_block();
                if (i + NS < nb && !*abort_flag) {
                    mbar_arrive_expect_tx(smem_u32(bars + slot), kBoxBytes);
                    tma_load_2d_hint(smem_u32(ring + slot * kBoxBytes), &a.tmW,
                                     (box0 + i + NS) * (kBoxCodes / 2), tile * kTile, smem_u32(bars + slot), pol);
                    last_box[slot] = i + NS;
                }
            }
        }
        if (++slot == NS) {
            slot = 0;
            ph ^= 1u;
        }
        const uint8_t* ab = act + i * kBoxAct;
        #pragma unroll
        for (int ci = 0; ci < CPT; ++ci) {
            const int c = t + TPR * ci;
            const uint8_t* ac = ab + c * kChunkAct;
            const uint32_t w[4] = {wv[ci].x, wv[ci].y, wv[ci].z, wv[ci].w};
            int lo[4], hi[4];
            #pragma unroll
            for (int j = 0; j < 4; ++j) {
                lo[j] = (int)((w[j] << 4) & 0xF0F0F0F0u);
                hi[j] = (int)(w[j] & 0xF0F0F0F0u);
            }
            #pragma unroll
            for (int m = 0; m < MT; ++m) {
                const uint4 a0 = *reinterpret_cast<const uint4*>(ac + m * 32);
                const uint4 a1 = *reinterpret_cast<const uint4*>(ac + m * 32 + 16);
                acc[m][0] = __dp4a(lo[0], (int)a0.x, acc[m][0]);
                acc[m][1] = __dp4a(hi[0], (int)a0.y, acc[m][1]);
                acc[m][0] = __dp4a(lo[1], (int)a0.z, acc[m][0]);
                acc[m][1] = __dp4a(hi[1], (int)a0.w, acc[m][1]);
                acc[m][0] = __dp4a(lo[2], (int)a1.x, acc[m][0]);
                acc[m][1] = __dp4a(hi[2], (int)a1.y, acc[m][1]);
                acc[m][0] = __dp4a(lo[3], (int)a1.z, acc[m][0]);
                acc[m][1] = __dp4a(hi[3], (int)a1.w, acc[m][1]);
            }
        }
    }

    // The row's sums (the two dp4a sums are 16 x integers); the warps of
    // chunk phases t > 0 hand theirs to phase 0, which adds them.
    int v[MT];
    #pragma unroll
    for (int m = 0; m < MT; ++m) v[m] = (acc[m][0] >> 4) + (acc[m][1] >> 4);
    if (t > 0) {
        #pragma unroll
        for (int m = 0; m < MT; ++m) red[((t - 1) * MT + m) * kTile + r] = v[m];
    }
    __syncthreads();
    if (*abort_flag && tid == 0) {
        // copies may still be landing after an abandoned wait: wait for the
        // last one of each slot (bounded) so none writes shared memory after exit
        if (!mbar_wait(smem_u32(bars + NS), 0)) atomicOr(&g_rowdot_error, kErrDrainWait);
        for (int s = 0; s < NS; ++s)
            if (last_box[s] >= 0 && !mbar_wait(smem_u32(bars + s), (uint32_t)(last_box[s] / NS) & 1u))
                atomicOr(&g_rowdot_error, kErrDrainWait);
    }
    if (t == 0) {
        #pragma unroll
        for (int tt = 1; tt < TPR; ++tt) {
            #pragma unroll
            for (int m = 0; m < MT; ++m) {
                v[m] += red[((tt - 1) * MT + m) * kTile + r];
            }
        }
    }
    const int n = tile * kTile + r;
    if (a.P == 1) {
        if (t == 0 && n < a.N) {
            const float swv = a.sw[n];
            #pragma unroll
            for (int m = 0; m < MT; ++m) {
                a.Y[(int64_t)m * a.N + n] = __fmul_rn(__fmul_rn(__int2float_rn(v[m]), swv), a.sa[m]);
                if (a.acc_out != nullptr) a.acc_out[(int64_t)m * a.N + n] = v[m];
            }
        }
        return;
    }

    // ------------------------------------------------ split K: last CTA sums
    if (t == 0) {
        int32_t* dst = a.part + ((int64_t)(tile * a.P + p) * MT) * kTile + r;
        #pragma unroll
        for (int m = 0; m < MT; ++m) dst[m * kTile] = v[m];
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) *last_flag = (atomicAdd(a.tickets + tile, 1u) == (unsigned)(a.P - 1));
    __syncthreads();
    if (!*last_flag) return;
    __threadfence();
    const int32_t* src = a.part + (int64_t)tile * a.P * MT * kTile;
    for (int e = tid; e < MT * kTile; e += kThreads) {
        const int m = e / kTile, rr = e % kTile, nn = tile * kTile + rr;
        if (nn >= a.N) continue;
        int32_t sum = 0;
        for (int q = 0; q < a.P; ++q) sum += __ldcg(src + (int64_t)q * MT * kTile + e);
        a.Y[(int64_t)m * a.N + nn] = __fmul_rn(__fmul_rn(__int2float_rn(sum), a.sw[nn]), a.sa[m]);
        if (a.acc_out != nullptr) a.acc_out[(int64_t)m * a.N + nn] = sum;
    }
    if (tid == 0) a.tickets[tile] = 0u;  // ready for the next call
}

// Group-wise scales (groups of gs = 2^gshift codes, 32 <= gs <= K): the
// order of the fp32 arithmetic is fixed by K and gs alone, so the result is
// the same bits whatever the launch plan:
//   acc_g = the exact int32 sum of group g,
//   per chunk of L = max(gs, 1024) codes: f = +0, then for its groups in
//   ascending order f = fma((float)acc_g, s_g, f),
//   T = +0, then for the chunks in ascending order T = T + f,
//   Y = T * s_a.
// Each chunk of a weight row is walked in K order by one thread, so its
// fold needs no exchange: a CTA has nph phases of 128 threads (one per
// weight row), phase h taking the piece's chunks h, h + nph, ...; each
// thread reads all eight 16-byte chunks of its row from every box of its
// chunks (the swizzle keeps a quarter-warp's eight lanes on eight bank
// groups).  A ring slot holds a box of weights and that box's activation
// codes ([8][MT][32 bytes], one bulk copy on the same mbarrier), so no
// piece length limit comes from the activations.  The chunk sums go to T
// in registers (one phase, one piece), to shared memory for phase 0 to add
// in chunk order (several phases, one piece), or to the workspace for the
// CTA that finishes a tile last (K split into pieces of whole chunks).
// The group scales are read from global memory one box ahead (prefetched
// into L1 for the whole piece).
template <int MT>
__global__ void __launch_bounds__(kTile * kMaxPhases, 1) rowdot_group_kernel(const __grid_constant__ GroupArgs a) {
    constexpr int kWarps = kTile / 32;  // warps of one phase
    constexpr int kChunkAct = MT * 32;
    constexpr int kBoxAct = 8 * kChunkAct;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const int NS = a.NS;
    const int cpp = a.bpp / a.abox;                                // chunks per piece
    uint8_t* ring = smem;                                          // [NS][16384] weights
    uint8_t* acts = smem + NS * kBoxBytes;                         // [NS][kBoxAct] codes
    float* cval = reinterpret_cast<float*>(acts + NS * kBoxAct);   // [MT][cpp][128] when nph > 1, P == 1
    uint64_t* bars = reinterpret_cast<uint64_t*>(cval + (a.nph > 1 && a.P == 1 ? MT * cpp * kTile : 0));
    int* released = reinterpret_cast<int*>(bars + NS);
    volatile int* last_box = released + NS;  // box of each slot's latest fill
    volatile int* abort_flag = last_box + NS;
    int* last_flag = const_cast<int*>(last_box) + NS + 1;

    const int tid = threadIdx.x, lane = tid & 31;
    const int r = tid & (kTile - 1);  // weight row within the tile
    const int ph = tid / kTile;       // phase: chunks ph, ph + nph, ... of the piece
    const int nph = a.nph;
    const int tg = blockIdx.x / a.P, p = blockIdx.x % a.P;  // tile of all matrices, K piece
    int g = 0;
    #pragma unroll
    for (int k = 1; k < kGroupMats; ++k) g += (tg >= a.tile0[k]) ? 1 : 0;
    const int tile = tg - a.tile0[g];  // tile within matrix g
    const CUtensorMap* tmW = &a.tmW[g];
    const int Ng = a.N[g];
    const int box0 = p * a.bpp;
    const int nb = min(a.bpp, a.nbox - box0);
    const uint64_t pol = l2_evict_first_policy();
    const uint64_t pol_act = l2_evict_last_policy();
    const uint8_t* codes = a.codes;
    const int64_t n = (int64_t)tile * kTile + r;
    const bool row_ok = n < Ng;
    const float* srow = a.sg[g] + (row_ok ? n : 0) * a.gld;
    const int gmask = (1 << a.gshift) - 1;
    const int lmask = (1 << a.lshift) - 1;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_u32(bars + s), 1);
            released[s] = 0;
            last_box[s] = -1;
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    griddep_launch_dependents();
    const int n0 = min(NS, nb);
    if (tid == 0) {  // the weights do not depend on earlier launches
        for (int i = 0; i < n0; ++i) {
            mbar_arrive_expect_tx(smem_u32(bars + i), kBoxBytes + kBoxAct);
            tma_load_2d_hint(smem_u32(ring + i * kBoxBytes), tmW, (box0 + i) * (kBoxCodes / 2),
                             tile * kTile, smem_u32(bars + i), pol);
            last_box[i] = i;
        }
    }
    // the boxes of this phase: i = abox * (chunk) + j for chunks ph, ph + nph, ...
    auto next_box = [&](int i) { return (i + 1) % a.abox ? i + 1 : i + 1 + (nph - 1) * a.abox; };
    // the row's scales for the piece into L1 (128-byte lines), so that the
    // loads one box ahead hit it
    if (ph == 0) {
        const int ga = min((box0 * kBoxCodes) >> a.gshift, a.ngroups - 1);
        const int gb = min(((box0 + nb) * kBoxCodes - 1) >> a.gshift, a.ngroups - 1);
        const uintptr_t lo = reinterpret_cast<uintptr_t>(srow + ga) & ~(uintptr_t)127;
        const uintptr_t hi = reinterpret_cast<uintptr_t>(srow + gb);
        for (uintptr_t q = lo; q <= hi; q += 128) prefetch_l1(reinterpret_cast<const void*>(q));
    }
    // scales of the groups that end in the 8 chunks of box i (rows past N
    // read row 0's and write nothing; chunks past K clamp to the last group).
    // Only a chunk that ends a group uses its scale: boxes start on 256-code
    // boundaries, so for groups of at most 256 codes that is every chunk
    // with 32 (c + 1) a multiple of the group, for longer groups at most the
    // last chunk (uniform over the CTA; 2 loads a box instead of 8 at
    // groups of 128 codes)
    auto load_scales = [&](int i, float* sc) {
        #pragma unroll
        for (int c = 0; c < 8; ++c) {
            if (((32 * (c + 1)) & gmask) == 0 || c == 7) {
                const int gi = min(((box0 + i) * kBoxCodes + 32 * c) >> a.gshift, a.ngroups - 1);
                sc[c] = __ldg(srow + gi);
            } else {
                sc[c] = 0.f;
            }
        }
    };
    const int i_first = ph * a.abox;
    float sc[8];
    load_scales(min(i_first, nb - 1), sc);
    griddep_wait();  // activation codes, outputs and workspace from here on
    if (tid == 0) {
        for (int i = 0; i < n0; ++i)
            bulk_g2s(smem_u32(acts + i * kBoxAct), codes + (int64_t)(box0 + i) * kBoxAct, kBoxAct,
                     smem_u32(bars + i), pol_act);
    }

    int acc[MT][2];  // 16 x the even / odd products of the current group
    float f[MT], T[MT];
    #pragma unroll
    for (int m = 0; m < MT; ++m) {
        acc[m][0] = acc[m][1] = 0;
        f[m] = 0.f;
        T[m] = 0.f;
    }
    const uint8_t* wrow = ring + r * 128;
    for (int i = i_first; i < nb; i = next_box(i)) {
        const int slot = i % NS;
        float scn[8];
        const int in = next_box(i);
        load_scales(in < nb ? in : i, scn);
        // the slot must hold box i's fill before its parity means anything;
        // warp-uniform outcome, so the warp's __syncwarp below never splits
        if (!__all_sync(0xFFFFFFFFu, wait_slot_box(last_box + slot, i, abort_flag) &&
                                         wait_bounded(smem_u32(bars + slot), (uint32_t)(i / NS) & 1u, abort_flag)))
            break;
        uint4 wv[8];
        #pragma unroll
        for (int c = 0; c < 8; ++c)
            wv[c] = *reinterpret_cast<const uint4*>(wrow + slot * kBoxBytes + ((c ^ (r & 7)) << 4));
        const uint8_t* ab = acts + slot * kBoxAct;
        const int pos = (box0 + i) * kBoxCodes;  // first code of the box
        #pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint8_t* ac = ab + c * kChunkAct;
            const uint32_t w[4] = {wv[c].x, wv[c].y, wv[c].z, wv[c].w};
            int lo[4], hi[4];
            #pragma unroll
            for (int j = 0; j < 4; ++j) {
                lo[j] = (int)((w[j] << 4) & 0xF0F0F0F0u);
                hi[j] = (int)(w[j] & 0xF0F0F0F0u);
            }
            #pragma unroll
            for (int m = 0; m < MT; ++m) {
                const uint4 a0 = *reinterpret_cast<const uint4*>(ac + m * 32);
                const uint4 a1 = *reinterpret_cast<const uint4*>(ac + m * 32 + 16);
                acc[m][0] = __dp4a(lo[0], (int)a0.x, acc[m][0]);
                acc[m][1] = __dp4a(hi[0], (int)a0.y, acc[m][1]);
                acc[m][0] = __dp4a(lo[1], (int)a0.z, acc[m][0]);
                acc[m][1] = __dp4a(hi[1], (int)a0.w, acc[m][1]);
                acc[m][0] = __dp4a(lo[2], (int)a1.x, acc[m][0]);
                acc[m][1] = __dp4a(hi[2], (int)a1.y, acc[m][1]);
                acc[m][0] = __dp4a(lo[3], (int)a1.z, acc[m][0]);
                acc[m][1] = __dp4a(hi[3], (int)a1.w, acc[m][1]);
            }
            const int end = pos + 32 * (c + 1);  // codes done after this chunk
            if ((end & gmask) == 0 && end <= a.K) {  // a group ends (uniform over the CTA)
                #pragma unroll
                for (int m = 0; m < MT; ++m) {
                    f[m] = __fmaf_rn(__int2float_rn((acc[m][0] >> 4) + (acc[m][1] >> 4)), sc[c], f[m]);
                    acc[m][0] = acc[m][1] = 0;
                }
                if ((end & lmask) == 0 || end == a.K) {  // so does a fold chunk
                    if (a.P == 1 && nph == 1) {
                        #pragma unroll
                        for (int m = 0; m < MT; ++m) T[m] = __fadd_rn(T[m], f[m]);
                    } else if (a.P == 1) {
                        const int cl = i / a.abox;  // chunk within the piece
                        #pragma unroll
                        for (int m = 0; m < MT; ++m) cval[(m * cpp + cl) * kTile + r] = f[m];
                    } else {
                        float* dst = a.part_f + ((int64_t)(tg * a.nch + ((end - 1) >> a.lshift)) * MT) * kTile + r;
                        #pragma unroll
                        for (int m = 0; m < MT; ++m) dst[m * kTile] = f[m];
                    }
                    #pragma unroll
                    for (int m = 0; m < MT; ++m) f[m] = 0.f;
                }
            }
        }
        #pragma unroll
        for (int c = 0; c < 8; ++c) sc[c] = scn[c];
        __syncwarp();
        if (lane == 0) {
            // the last of the phase's warps done with this slot (weights and
            // codes) refills it with the box NS further on
            __threadfence_block();
            if (atomicAdd(released + slot, 1) == kWarps - 1) {
                released[slot] = 0;
                __threadfence_block();
                if (i + NS < nb && !*abort_flag) {
                    const uint32_t bar = smem_u32(bars + slot);
                    mbar_arrive_expect_tx(bar, kBoxBytes + kBoxAct);
                    tma_load_2d_hint(smem_u32(ring + slot * kBoxBytes), tmW, (box0 + i + NS) * (kBoxCodes / 2),
                                     tile * kTile, bar, pol);
                    bulk_g2s(smem_u32(acts + slot * kBoxAct), codes + (int64_t)(box0 + i + NS) * kBoxAct, kBoxAct,
                             bar, pol_act);
                    last_box[slot] = i + NS;  // box i's fill is consumed: the parity now tracks box i + NS
                    __threadfence_block();
                }
            }
        }
    }

    __syncthreads();
    if (*abort_flag && tid == 0) {
        // copies may still be landing after an abandoned wait: wait for the
        // last one of each slot (bounded) so none writes shared memory after exit
        for (int s = 0; s < NS; ++s)
            if (last_box[s] >= 0 && !mbar_wait(smem_u32(bars + s), (uint32_t)(last_box[s] / NS) & 1u))
                atomicOr(&g_rowdot_error, kErrDrainWait);
    }
    if (*abort_flag) return;
    float* Y = a.Y[g];
    if (a.P == 1) {
        if (ph == 0 && row_ok) {
            #pragma unroll
            for (int m = 0; m < MT; ++m) {
                float t = T[m];
                if (nph > 1) {  // the phases' chunk sums, in chunk order
                    t = 0.f;
                    for (int cl = 0; cl < cpp; ++cl) t = __fadd_rn(t, cval[(m * cpp + cl) * kTile + r]);
                }
                Y[(int64_t)m * Ng + n] = __fmul_rn(t, a.sa[m]);
            }
        }
        return;
    }

    // ------------------------------------ split K: the last CTA adds the chunks
    __threadfence();
    __syncthreads();
    if (tid == 0) *last_flag = (atomicAdd(a.tickets + tg, 1u) == (unsigned)(a.P - 1));
    __syncthreads();
    if (!*last_flag) return;
    __threadfence();
    if (ph == 0 && row_ok) {
        // chunk sums in chunk order; loads issued 8 at a time ahead of the adds
        const float* src = a.part_f + (int64_t)tg * a.nch * MT * kTile + r;
        #pragma unroll
        for (int m = 0; m < MT; ++m) {
            float t = 0.f;
            for (int c0 = 0; c0 < a.nch; c0 += 8) {
                float v[8];
                #pragma unroll
                for (int k = 0; k < 8; ++k)
                    v[k] = c0 + k < a.nch ? __ldcg(src + ((int64_t)(c0 + k) * MT + m) * kTile) : 0.f;
                #pragma unroll
                for (int k = 0; k < 8; ++k)
                    if (c0 + k < a.nch) t = __fadd_rn(t, v[k]);
            }
            Y[(int64_t)m * Ng + n] = __fmul_rn(t, a.sa[m]);
        }
    }
    if (tid == 0) a.tickets[tg] = 0u;  // ready for the next call
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

template <int MT, int TPR>
const void* kernel_for() {
    return reinterpret_cast<const void*>(rowdot_kernel<MT, TPR>);
}

template <int TPR>
const void* kernel_for_rows(int M) {
    switch (M) {
        case 2: return kernel_for<2, TPR>();
        case 3: return kernel_for<3, TPR>();
        case 4: return kernel_for<4, TPR>();
        case 5: return kernel_for<5, TPR>();
        case 6: return kernel_for<6, TPR>();
        case 7: return kernel_for<7, TPR>();
        case 8: return kernel_for<8, TPR>();
        default: return nullptr;
    }
}

const void* group_kernel_for(int M) {
    switch (M) {
        case 1: return reinterpret_cast<const void*>(rowdot_group_kernel<1>);
        case 2: return reinterpret_cast<const void*>(rowdot_group_kernel<2>);
        case 3: return reinterpret_cast<const void*>(rowdot_group_kernel<3>);
        case 4: return reinterpret_cast<const void*>(rowdot_group_kernel<4>);
        case 5: return reinterpret_cast<const void*>(rowdot_group_kernel<5>);
        case 6: return reinterpret_cast<const void*>(rowdot_group_kernel<6>);
        case 7: return reinterpret_cast<const void*>(rowdot_group_kernel<7>);
        case 8: return reinterpret_cast<const void*>(rowdot_group_kernel<8>);
        default: return nullptr;
    }
}

// Row-wise scales: 2, 4 or 8 threads per row; group scales: 1, 2 or 4
// phases (one kernel).
const void* kernel_for(int M, int tpr, bool group) {
    if (group) return (tpr == 1 || tpr == 2 || tpr == 4) ? group_kernel_for(M) : nullptr;
    switch (tpr) {
        case 2: return kernel_for_rows<2>(M);
        case 4: return kernel_for_rows<4>(M);
        case 8: return kernel_for_rows<8>(M);
        default: return nullptr;
    }
}

// Opts every instantiation into its largest shared-memory plan (and the
// full shared-memory carveout, so that the planned CTAs per SM fit), once
// per device.
cudaError_t set_attributes() {
    static bool done[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && done[dev]) return cudaSuccess;
    for (int k = 0; k < 4; ++k) {
        for (int M = 1; M <= kRowdotMaxM; ++M) {
            const void* fn = k < 3 ? kernel_for(M, 2 << k, false) : kernel_for(M, 1, true);
            if (fn == nullptr) continue;
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemPerSM - 1024);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
            if (e != cudaSuccess) return e;
        }
    }
    if (dev < 64) done[dev] = true;
    return cudaSuccess;
}

size_t smem_bytes(int M, int NS, int bpp, int tpr) {
    return 1024 + (size_t)NS * kBoxBytes + (size_t)M * bpp * kActBoxBytes +
           (size_t)(tpr - 1) * M * kTile * 4 + (size_t)(NS + 1) * 8 + (size_t)(2 * NS + 2) * 4;
}

// Group-scale kernel: NS slots of one weight box and its activation codes,
// and cval_bytes of chunk sums.
size_t group_smem_bytes(int M, int NS, size_t cval_bytes) {
    return 1024 + (size_t)NS * (kBoxBytes + (size_t)M * kActBoxBytes) + cval_bytes + (size_t)NS * 8 +
           (size_t)(2 * NS + 2) * 4;
}

constexpr int kMaxNSGroup = 16;

// Group scales (groups of 2^gshift codes): 1..8 batch rows, phases of 128
// threads (one per weight row).  K is split into pieces of whole chunks
// (max(group, 1024) codes) while the tiles cover less than 4/5 of the SMs
// (or into min(force_p, chunks) pieces when force_p > 0); then as many CTAs
// per SM as the grid fills (at most 4, or cps when given), 4 / cps phases
// per CTA (at most one per chunk of a piece), and the ring takes the shared
// memory left, so that every SM keeps 16 warps and about 12 boxes in flight.  N counts
// the rows of all matrices of a launch (each padded to whole tiles by the
// caller when the plan is for a launch, or the sum of the rows for the
// workspace bound, which then covers kGroupMats - 1 partial tiles more).
bool make_group_plan(int M, int64_t K, int64_t N, int num_sms, RowdotPlan* out, int cps, int gshift,
                     int force_p) {
    if (M < 1 || M > kRowdotMaxM || K < 32 || K % 32 || K > 131072 || N < 1 || N > 0x7FFFFFFF)
        return false;
    if (gshift < 5 || gshift > 17 || K % (1LL << gshift)) return false;
    if (cps < 0 || cps > 4 || num_sms < 1) return false;
    RowdotPlan pl = {};
    pl.tpr = 1;
    pl.MT = M;
    pl.force_p = force_p;
    pl.cps_req = cps;
    pl.gshift = gshift;
    pl.lshift = gshift > 10 ? gshift : 10;
    pl.tiles = (int)((N + kTile - 1) / kTile);
    pl.nbox = (int)((K + kBoxCodes - 1) / kBoxCodes);
    pl.nch = (int)((K + (1LL << pl.lshift) - 1) >> pl.lshift);
    const int abox = (1 << pl.lshift) / kBoxCodes;  // boxes per chunk
    // split while the tiles cover less than 4/5 of the SMs
    int P = (num_sms * 4 / 5 + pl.tiles - 1) / pl.tiles;
    if (force_p > 0) P = force_p;
    if (P > pl.nch) P = pl.nch;
    if (P < 1 || pl.tiles > kTicketSlots) P = 1;  // one arrival counter per tile
    const int cpp = (pl.nch + P - 1) / P;  // chunks per piece
    pl.P = (pl.nch + cpp - 1) / cpp;
    pl.bpp = cpp * abox;
    if ((int64_t)pl.tiles * pl.P > 0x7FFFFFFF) return false;
    const int64_t ctas = (int64_t)pl.tiles * pl.P;
    pl.cps = cps > 0 ? cps : (int)((ctas + num_sms - 1) / num_sms < 4 ? (ctas + num_sms - 1) / num_sms : 4);
    pl.abox = abox;
    int nph = kMaxPhases / pl.cps;
    while (nph > cpp) nph /= 2;
    size_t cval = (nph > 1 && pl.P == 1) ? (size_t)M * cpp * kTile * 4 : 0;
    if (cval > 32 * 1024) {  // chunk sums of a long row: one phase keeps them in registers
        nph = 1;
        cval = 0;
    }
    pl.nph = nph;
    pl.tpr = nph;
    const int budget = kSmemPerSM / pl.cps - 1024;
    int NS = kMaxNSGroup;
    while (NS > 1 && group_smem_bytes(M, NS, cval) > (size_t)budget) --NS;
    if (group_smem_bytes(M, NS, cval) > (size_t)budget) return false;
    pl.NS = NS;
    pl.smem = (int)group_smem_bytes(M, NS, cval);
    pl.grid = (int)ctas;
    pl.sms = num_sms;
    // workspace: tickets, scales, activation codes [nbox][8][M][32 bytes],
    // then chunk sums [tiles][nch][M][128] fp32.  K is split only when the
    // tiles are fewer than the SMs (or on request), and a launch of several
    // matrices has at most kGroupMats - 1 tiles more than their summed rows.
    pl.off_sa = kTicketBytes;
    pl.off_codes = pl.off_sa + 256;
    pl.off_part = round_up_sz(pl.off_codes + (size_t)M * pl.nbox * kActBoxBytes, 256);
    int64_t tmax = 0;
    if (pl.nch > 1) {
        tmax = pl.tiles + kGroupMats - 1;
        if (force_p <= 1 && tmax > num_sms * 4 / 5) tmax = num_sms * 4 / 5;
    }
    pl.ws_bytes = pl.off_part + round_up_sz((size_t)tmax * pl.nch * M * kTile * 4, 256);
    *out = pl;
    return true;
}

}  // namespace

// Plan: one CTA per 128 weight rows and K piece, TPR threads per row and
// cps CTAs per SM (0 = the defaults: 4 threads, 4 / TPR CTAs).  K is split
// into pieces of whole 256-code boxes when the tiles alone leave CTA slots
// idle, and so that a piece's activation codes fit in kActMax bytes.  The
// ring takes what shared memory is left, up to kMaxNS boxes.  gshift >= 0:
// group scales (groups of 2^gshift codes), the one-thread-per-row kernel.
bool make_rowdot_plan(int M, int64_t K, int64_t N, int num_sms, RowdotPlan* out, int tpr, int cps,
                      int gshift, int force_p) {
    if (gshift >= 0) return make_group_plan(M, K, N, num_sms, out, cps, gshift, force_p);
    if (M < 2 || M > kRowdotMaxM || K < 32 || K % 32 || K > 131072 || N < 1 || N > 0x7FFFFFFF)
        return false;
    if (tpr == 0) tpr = kRowdotDefaultTPR;
    if (tpr != 2 && tpr != 4 && tpr != 8) return false;
    if (cps == 0) cps = tpr < 4 ? 4 / tpr : 1;
    if (cps < 1 || cps > 4) return false;
    RowdotPlan pl = {};
    pl.tpr = tpr;
    pl.MT = M;
    pl.tiles = (int)((N + kTile - 1) / kTile);
    pl.nbox = (int)((K + kBoxCodes - 1) / kBoxCodes);
    pl.cps = cps;
    const int slots = pl.cps * num_sms;
    int P = 1;
    if (pl.tiles < slots * 4 / 5) P = slots / pl.tiles;
    const int bpp_max = kActMax / (M * kActBoxBytes);
    const int pmin = (pl.nbox + bpp_max - 1) / bpp_max;
    if (P < pmin) P = pmin;
    if (P > pl.nbox) P = pl.nbox;
    pl.bpp = (pl.nbox + P - 1) / P;
    pl.P = (pl.nbox + pl.bpp - 1) / pl.bpp;
    if (pl.P > 1 && pl.tiles > kTicketSlots) return false;
    if ((int64_t)pl.tiles * pl.P > 0x7FFFFFFF) return false;
    pl.gshift = -1;
    const int budget = kSmemPerSM / pl.cps - 1024;
    int NS = kMaxNS < pl.bpp ? kMaxNS : pl.bpp;
    while (NS > 1 && smem_bytes(M, NS, pl.bpp, tpr) > (size_t)budget) --NS;
    if (smem_bytes(M, NS, pl.bpp, tpr) > (size_t)budget) return false;
    pl.NS = NS;
    pl.smem = (int)smem_bytes(M, NS, pl.bpp, tpr);
    pl.grid = pl.tiles * pl.P;
    pl.sms = num_sms;
    // workspace: tickets, scales, activation codes [nbox][8][M][32 bytes],
    // then piece sums [tiles][P][M][128] int32.
    // Sized for any N' <= N (grouped launches plan each matrix on its own):
    // a matrix is split either because its tiles leave CTA slots idle
    // (then tiles' * P' <= slots) or because a piece's codes must fit in
    // kActMax (P' = pmin, tiles' <= tiles), so max(slots, tiles * pmin)
    // tile pieces when pmin > 1, else slots.
    pl.off_sa = kTicketBytes;
    pl.off_codes = pl.off_sa + 256;
    pl.off_part = round_up_sz(pl.off_codes + (size_t)M * pl.nbox * kActBoxBytes, 256);
    int64_t units = slots;
    if (pmin > 1 && units < (int64_t)pl.tiles * pmin) units = (int64_t)pl.tiles * pmin;
    if (pl.P > 1 && units < (int64_t)pl.tiles * pl.P) units = (int64_t)pl.tiles * pl.P;
    pl.ws_bytes = pl.off_part + round_up_sz((size_t)units * M * kTile * 4, 256);
    *out = pl;
    return true;
}

cudaError_t launch_w4a8_rowdot(const RowdotPlan& pl, const uint16_t* X, const int8_t* Xq,
                               const float* sa, int M, int64_t K, int G, const uint8_t* const* Wq,
                               const float* const* sw, const int64_t* Ns, float* const* Y,
                               int32_t* acc_out, int8_t* Xq_out, float* sa_out, void* ws,
                               unsigned flags, cudaStream_t stream, int gs, const float* const* sg) {
    const bool group = gs > 0;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    float* sa_ws = reinterpret_cast<float*>(wsb + pl.off_sa);
    uint2* codes = reinterpret_cast<uint2*>(wsb + pl.off_codes);
    const int64_t kw = (int64_t)pl.nbox * (kBoxCodes / 8);
    {
        const __half* xh = reinterpret_cast<const __half*>(X);
        int Mi = M;
        int64_t Kk = K, kwv = kw;
        void* args[] = {&xh, &Xq, &sa, &Mi, &Kk, &kwv, &codes, &sa_ws, &Xq_out, &sa_out};
        const unsigned pieces = (unsigned)((kw + kPreThreads - 1) / kPreThreads);
        cudaError_t e = launch_pdl(reinterpret_cast<const void*>(rowdot_codes_kernel), dim3(M, pieces),
                                   dim3(kPreThreads), 0, stream, flags, args);
        if (e != cudaSuccess) return e;
    }
    const void* fn = kernel_for(M, pl.tpr, group);
    if (fn == nullptr || group != (pl.gshift >= 0)) return cudaErrorInvalidValue;
    cudaError_t e = set_attributes();
    if (e != cudaSuccess) return e;
    if (group) {
        // every matrix in one launch, their tiles numbered consecutively
        if (G < 1 || G > kGroupMats) return cudaErrorInvalidValue;
        GroupArgs a;
        memset(&a, 0, sizeof(a));
        int64_t tiles = 0;
        for (int g = 0; g < G; ++g) {
            if (!make_w4_tile_map(&a.tmW[g], Wq[g], K, Ns[g])) return cudaErrorInvalidValue;
            a.sg[g] = sg[g];
            a.Y[g] = Y[g];
            a.N[g] = (int)Ns[g];
            a.tile0[g] = (int)tiles;
            tiles += (Ns[g] + kTile - 1) / kTile;
        }
        for (int g = G; g <= kGroupMats; ++g) a.tile0[g] = (int)tiles;
        RowdotPlan pg;
        if (!make_group_plan(M, K, tiles * kTile, pl.sms, &pg, pl.cps_req, pl.gshift, pl.force_p))
            return cudaErrorInvalidValue;
        // the caller's workspace (planned for the summed rows) holds this launch's chunk sums
        if (pg.off_part != pl.off_part ||
            pl.off_part + (pg.P > 1 ? (size_t)tiles * pg.nch * M * kTile * 4 : 0) > pl.ws_bytes)
            return cudaErrorInvalidValue;
        a.codes = reinterpret_cast<const uint8_t*>(codes);
        a.sa = sa_ws;
        a.part_f = reinterpret_cast<float*>(wsb + pg.off_part);
        a.tickets = reinterpret_cast<unsigned*>(wsb);
        a.gshift = pg.gshift;
        a.gld = (int)((K / gs + 3) / 4 * 4);
        a.ngroups = (int)(K >> pg.gshift);
        a.lshift = pg.lshift;
        a.nch = pg.nch;
        a.abox = pg.abox;
        a.K = (int)K;
        a.M = M;
        a.nbox = pg.nbox;
        a.bpp = pg.bpp;
        a.P = pg.P;
        a.NS = pg.NS;
        a.nph = pg.nph;
        void* args[] = {&a};
        return launch_pdl(fn, dim3(pg.grid), dim3(kTile * pg.nph), pg.smem, stream, flags, args);
    }
    for (int g = 0; g < G; ++g) {
        RowdotPlan pg;
        if (!make_rowdot_plan(M, K, Ns[g], pl.sms, &pg, pl.tpr, pl.cps, pl.gshift, pl.force_p))
            return cudaErrorInvalidValue;
        RowdotArgs a;
        memset(&a, 0, sizeof(a));
        if (!make_w4_tile_map(&a.tmW, Wq[g], K, Ns[g])) return cudaErrorInvalidValue;
        a.codes = codes;
        a.sw = sw[g];
        a.sa = sa_ws;
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
        void* args[] = {&a};
        e = launch_pdl(fn, dim3(pg.grid), dim3(kTile * pg.tpr), pg.smem, stream, flags, args);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t read_and_clear_rowdot_error(unsigned* flags, cudaStream_t stream) {
    unsigned v = 0, z = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_rowdot_error, sizeof(v), 0, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbolAsync(g_rowdot_error, &z, sizeof(z), 0, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    *flags |= v;
    return e;
}

}  // namespace w4a8
