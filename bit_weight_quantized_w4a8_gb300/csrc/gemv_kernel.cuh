// gemv_kernel.cuh -- the streaming weight-quantized GEMV kernel for sm_103a
// (included by the translation units that instantiate and launch it).
//
// W4A8 (the Jetson INT4 page, sections 正确方向 / 当前实现方式): INT4 codes
// are widened to int8 lanes in registers and multiplied against INT8
// activation codes with __dp4a into int32; y = ((float)acc * s_w) * s_a.
// W8A16 (the TPU-MLIR W8A16 page, section 4): INT8 codes are widened to
// binary16 exactly in registers and multiplied with the F16 activation by
// f16 x f16 -> f32 FMAs (exact products, fp32 sums); the per-channel scale
// multiplies the fp32 sum once.
//
// Both are HBM-bound at decode batch sizes, so the kernel is built around
// the weight stream (the W8A16 page's load/compute overlap, done with the
// TMA unit and an mbarrier ring instead of GDMA/BDC ping-pong):
//  * one producer warp issues 1-D bulk copies (cp.async.bulk, L2
//    evict-first) of whole rows, or of row-pieces when K is split, into an
//    NS-stage shared-memory ring; `full`/`empty` mbarriers hand stages over;
//  * 8 consumer warps: thread j of a row-piece owns granule columns
//    j, j+Cl, ...; its activation operands are loaded once into registers,
//    so shared memory traffic per weight byte is one write (TMA) + one read;
//  * int32 partial sums are shifted right by 4 (the nibble trick below
//    yields 16 * product) and reduced with warp shuffles, across warps in
//    shared memory when a row-piece spans several warps;
//  * split-K: int32 (or fp32) partials go to the workspace; the last CTA of
//    a row block (atomic ticket) sums them in a fixed order and rescales
//    once, so W4A8 stays bit-exact and W8A16 deterministic;
//  * programmatic dependent launch: weights are streamed before the wait
//    on the previous kernel; activations, outputs and workspace after it.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "kernels.h"
#include "plan.h"
#include "actq.cuh"
#include "ptx.cuh"
#include "silu.cuh"

namespace w4a8 {

// Device error word of the including translation unit (bounded waits that
// ran out); each unit reads and clears its own copy.
static __device__ unsigned g_device_error;

constexpr int kMaxSegments = 4;

struct GemvArgs {
    // Up to kMaxSegments weight matrices sharing the activation; their rows
    // are concatenated: segment g holds rows off[g] .. off[g+1]-1 of N.
    const uint8_t* W[kMaxSegments];   // W4: [N_g][K/2] packed nibbles; W8: [N_g][K] int8
    const void* wscale[kMaxSegments]; // W4: float[N_g]; W8: binary16[N_g]
    float* Yg[kMaxSegments];          // [M][N_g]
    int64_t off[kMaxSegments + 1];    // segment row offsets; off[G..] = N
    const int8_t* Xq;       // W4 unfused: [M][K] int8 codes
    const float* sa;        // W4 unfused: [M] activation scales
    const __half* X;        // W4 fused and W8: [M][K] binary16 activation
    int32_t* acc_out;       // optional [M][N] (W4, one segment)
    int8_t* Xq_out;         // optional [M][K] (W4 fused)
    float* sa_out;          // optional [M] (W4 fused)
    __half* H;              // optional [M][N/2] (W4, one segment of paired rows: row 2i is
                            // gate i, row 2i + 1 up i): H[m][i] = binary16(silu(Y[m][2i]) * Y[m][2i+1]);
                            // every CTA then owns whole pairs
    void* part;             // split partials [P][M][N] (int32 or fp32)
    const uint8_t* pf;      // optional: bytes [pf, pf + pf_bytes) of the next launch's
    int64_t pf_bytes;       // weights to bring into L2 (a multiple of 16; 0 = none),
    int64_t pf_share;       // pf_share bytes per CTA (a multiple of 16)
    unsigned* tickets;      // [Gs] arrival counters at the workspace start,
                            // zero between calls
    int M;
    int K;
    int N;
    GemvPlan pl;
};

// Gated products of the rows row0 .. row0 + nrows - 1 (whole pairs) of a
// paired-row call, from the outputs the CTA has just written.
__device__ __forceinline__ void silu_pairs(const GemvArgs& a, int64_t row0, int nrows, int tid) {
    const int np = nrows >> 1;
    const int64_t N = a.N;
    for (int q = tid; q < a.M * np; q += kConsumers) {
        const int m = q / np, i = q - m * np;
        const int64_t n = row0 + 2 * i;
        const float* y = a.Yg[0] + (int64_t)m * N + n;
        a.H[(int64_t)m * (N / 2) + (n >> 1)] = silu_mul_h(__ldcg(y), __ldcg(y + 1));
    }
}

// Waits on an mbarrier phase unless the CTA has already given up.  On a
// timeout it records `bit` in the device error word and tells the other
// threads (through `abort_flag`) to stop waiting; the caller carries on
// without valid data so every thread still meets every named barrier.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag, unsigned bit) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
        #pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            atomicOr(&g_device_error, bit);
            return false;
        }
    }
}

__device__ __forceinline__ float warp_max(float v) {
    #pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// max |x| over 8 binary16 values, as binary16 pairs (comparisons are exact).
__device__ __forceinline__ __half2 absmax8(uint4 h, __half2 m) {
    const __half2* p = reinterpret_cast<const __half2*>(&h);
    #pragma unroll
    for (int t = 0; t < 4; ++t) m = __hmax2(m, __habs2(p[t]));
    return m;
}

// 32 activation codes in natural order (two 16-byte words) -> the lane order
// of the packed weights: word t of a granule holds codes 8t..8t+7 with even
// k in the low nibbles and odd k in the high nibbles, so the even codes
// go to act[t] and the odd codes to act[4 + t].
__device__ __forceinline__ void permute_act(uint4 lo, uint4 hi, uint32_t* act) {
    const uint32_t n[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    #pragma unroll
    for (int t = 0; t < 4; ++t) {
        act[t] = __byte_perm(n[2 * t], n[2 * t + 1], 0x6420);
        act[4 + t] = __byte_perm(n[2 * t], n[2 * t + 1], 0x7531);
    }
}

// c0 += lo(q) * lo(x), c1 += hi(q) * hi(x): binary16 products, exact in
// fp32, accumulated in fp32 (one instruction each, at the FFMA rate).
__device__ __forceinline__ void fma_f16_f32x2(float& c0, float& c1, uint32_t q, uint32_t x) {
    asm("{\n\t.reg .f16 ql, qh, xl, xh;\n\t"
        "mov.b32 {ql, qh}, %2;\n\t"
        "mov.b32 {xl, xh}, %3;\n\t"
        "fma.rn.f32.f16 %0, ql, xl, %0;\n\t"
        "fma.rn.f32.f16 %1, qh, xh, %1;\n\t}"
        : "+f"(c0), "+f"(c1)
        : "r"(q), "r"(x));
}

__device__ __forceinline__ int segment_of(const GemvArgs& a, int64_t n) {
    int g = 0;
    #pragma unroll
    for (int k = 1; k < kMaxSegments; ++k) g += (n >= a.off[k]) ? 1 : 0;
    return g;
}

// Stage `st` of a CTA's weight stream (rows row0 + st * Rl ...) into ring
// slot `slot`: one 1-D bulk copy per run of whole rows, cut where a segment
// ends, or one copy per row-piece when K is split.  (Inlined: a call on the
// refill path costs register spills and delays the refill.)
__device__ __forceinline__ void issue_stage(const GemvArgs& a, uint8_t* smem, int st, int slot,
                                         int64_t row0, int nrows, int g0, uint64_t pol) {
    const GemvPlan& pl = a.pl;
    const int gp = min(pl.Gq, pl.Gt - g0);
    const int RBp = gp * kGranBytes;  // bytes of one row-piece
    const int64_t RB = (int64_t)pl.Gt * kGranBytes;
    const int r0 = st * pl.Rl;
    const int nr = min(pl.Rl, nrows - r0);
    const uint32_t dst = smem_u32(smem + slot * pl.stage_stride);
    const uint32_t bar = smem_u32(smem + pl.off_bars + 8 * slot);
    mbar_arrive_expect_tx(bar, (uint32_t)(nr * RBp));
    int64_t n = row0 + r0;
    const int64_t n_end = n + nr;
    while (n < n_end) {
        const int sg = segment_of(a, n);
        const int64_t run = min(n_end, a.off[sg + 1]) - n;
        const uint8_t* src = a.W[sg] + (n - a.off[sg]) * RB + (int64_t)g0 * kGranBytes;
        const uint32_t d = dst + (uint32_t)((n - row0 - r0) * RBp);
        if (pl.P == 1) {
            bulk_g2s(d, src, (uint32_t)(run * RBp), bar, pol);
        } else {
            for (int r = 0; r < run; ++r)
                bulk_g2s(d + r * RBp, src + (int64_t)r * RB, (uint32_t)RBp, bar, pol);
        }
        n += run;
    }
}

// SMAX bounds the granule columns per thread; kExactS says the plan uses
// exactly SMAX of them (no per-column test in the loop).
template <bool kW4, int MT, int SMAX, bool kFused, bool kExactS>
__global__ void __launch_bounds__(kThreads, MT == 1 ? 2 : 1) gemv_kernel(const __grid_constant__ GemvArgs a) {
    using AccT = typename std::conditional<kW4, int, float>::type;
    constexpr int kActWords = 8;  // registers per granule per activation row (W8: binary16 pairs)

    extern __shared__ __align__(1024) uint8_t smem[];
    const GemvPlan& pl = a.pl;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int p = blockIdx.x % pl.P;
    const int rb = blockIdx.x / pl.P;
    const int64_t N = a.N;
    // paired rows (H): whole pairs per CTA, so that its epilogue sees both rows
    const int64_t row0 = a.H ? 2 * ((int64_t)rb * (N / 2) / pl.Gs) : (int64_t)rb * N / pl.Gs;
    const int nrows = (int)((a.H ? 2 * ((int64_t)(rb + 1) * (N / 2) / pl.Gs) : (int64_t)(rb + 1) * N / pl.Gs) -
                            row0);
    const int nstages = (nrows + pl.Rl - 1) / pl.Rl;
    const int NS = pl.NS;
    const int g0 = p * pl.Gq;                   // first granule of this piece
    const int gp = min(pl.Gq, pl.Gt - g0);      // granules in this piece
    const int RBp = gp * kGranBytes;            // bytes of one row-piece

    uint64_t* full = reinterpret_cast<uint64_t*>(smem + pl.off_bars);
    uint64_t* sw_bar = full + NS;                       // scale cache landed
    int* released = reinterpret_cast<int*>(sw_bar + 1);  // warps done with each slot
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + pl.off_flag);
    int* last_flag = reinterpret_cast<int*>(smem + pl.off_flag + 4);
    float* sw_s = reinterpret_cast<float*>(smem + pl.off_sw);

    const uint64_t pol = l2_evict_first_policy();
    auto issue = [&](int st, int slot) { issue_stage(a, smem, st, slot, row0, nrows, g0, pol); };

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_u32(full + s), 1);
            released[s] = 0;
        }
        mbar_init(smem_u32(sw_bar), kConsumers);
        *abort_flag = 0;
        fence_mbar_init();
        // Fill the ring (weights may be read before the dependency wait).
        for (int st = 0; st < min(NS, nstages); ++st) issue(st, st);
        // The next launch's first weight bytes into L2, this CTA's share: at
        // one row the launch is latency-bound and leaves HBM idle meanwhile.
        if (a.pf_bytes > 0) {
            const int64_t o1 = min((int64_t)(blockIdx.x + 1) * a.pf_share, a.pf_bytes);
            for (int64_t o = (int64_t)blockIdx.x * a.pf_share; o < o1; o += 65536)
                prefetch_bulk_l2(a.pf + o, (uint32_t)min((int64_t)65536, o1 - o));
        }
    }
    griddep_launch_dependents();
    // Warm the L2 with the activation lines: a prefetch binds no value, so
    // it is safe before the dependency wait even if the previous kernel
    // is still writing them.
    {
        const void* xp = (kW4 && !kFused) ? static_cast<const void*>(a.Xq) : static_cast<const void*>(a.X);
        const int64_t xbytes = (int64_t)a.M * a.K * ((kW4 && !kFused) ? 1 : 2);
        for (int64_t o = (int64_t)threadIdx.x * 128; o < xbytes; o += (int64_t)kThreads * 128)
            prefetch_l2(static_cast<const uint8_t*>(xp) + o);
    }

    const int Cl = pl.Cl;
    const int i = tid >> pl.log2Cl;   // row-piece within a stage
    const int j = tid & (Cl - 1);     // column slot within the row-piece
    const int M = a.M;
    const int64_t K = a.K;
    // granule columns j, j+Cl, ... below gp belong to this thread
    const int ncol = j < gp ? min(pl.S, (gp - j + Cl - 1) >> pl.log2Cl) : 0;

    __syncthreads();  // barrier init visible to every thread
    // Weight scales of this CTA's rows (weights may be read before the wait):
    // asynchronous 4-byte copies whose completion arrives on sw_bar; only the
    // threads that write outputs wait for it, right before their first one.
    if constexpr (kW4) {
        if (pl.P == 1)
            for (int r = tid; r < nrows; r += kConsumers)
            {
                const int64_t n = row0 + r;
                const int sg = segment_of(a, n);
                cp_async_4(smem_u32(sw_s + r), static_cast<const float*>(a.wscale[sg]) + (n - a.off[sg]));
            }
        cp_async_mbar_arrive(smem_u32(sw_bar));
    } else {
        // binary16 scales (one segment): the 4-byte words covering rows
        // row0 & ~1 ... row0 + nrows - 1; a word past the last scale reads
        // only its first half
        if (pl.P == 1) {
            const uint16_t* s16 = static_cast<const uint16_t*>(a.wscale[0]);
            const int64_t base = row0 & ~(int64_t)1;
            const int words = (int)((row0 + nrows - base + 1) >> 1);
            for (int w = tid; w < words; w += kConsumers) {
                const int64_t e = base + 2 * w;
                cp_async_4_partial(smem_u32(sw_s + w), s16 + e, e + 1 < N ? 4u : 2u);
            }
        }
        cp_async_mbar_arrive(smem_u32(sw_bar));
    }

    griddep_wait();  // activations, outputs and workspace from here on

    uint32_t act[MT][SMAX][kActWords];
    float sa_r[MT];

    if constexpr (kW4 && kFused) {
        // Dynamic activation quantization fused into the linear (the Jetson
        // INT4 page, section 后续优化方向).  Every CTA derives the same s_a
        // from the whole row, then quantizes only its own K piece into
        // shared memory, already in the lane order of the packed weights:
        // per row piece, plane 0 holds granule c's even-k codes as 16 bytes
        // at 16c, plane 1 its odd-k codes at 16 (Gq + c), so that threads of
        // consecutive columns read consecutive 16-byte words.
        float* max_s = reinterpret_cast<float*>(smem + pl.off_max);
        uint32_t* act_w = reinterpret_cast<uint32_t*>(smem + pl.off_act);
        const int act_words = pl.Gq * 8;       // words per activation row piece
        const int plane = pl.Gq * 4;           // words per plane
        const int nv = (int)(K / 8);           // 16-byte vectors per activation row
        const int v0 = g0 * 4;                 // first vector of this piece
        const int nvq = gp * 4;                // vectors in this piece
        uint4* x_s = reinterpret_cast<uint4*>(smem + pl.off_x);
        // vector v of the piece = codes 8t..8t+7 of granule v / 4: its even
        // codes are word v of plane 0, its odd codes word v of plane 1
        auto quant_piece = [&](const uint4* src, uint32_t* dst, float sa, float r_lo, float r_hi) {
            #pragma unroll 2
            for (int v = tid; v < nvq; v += kConsumers) {
                const uint2 q = quant8_split(src[v], sa, r_lo, r_hi);
                dst[v] = q.x;
                dst[plane + v] = q.y;
            }
        };
        const bool staged = MT == 1 && pl.x_bytes > 0;
        if (staged) {
            // M == 1, short row: every thread copies its 16-byte vectors to
            // shared memory asynchronously (all in flight at once), then
            // takes the max over the vectors it copied
            const uint4* xv = reinterpret_cast<const uint4*>(a.X);
            #pragma unroll 1
            for (int v = tid; v < nv; v += kConsumers) cp_async_16(smem_u32(x_s + v), xv + v);
            cp_async_wait_all();
            __half2 hm = __float2half2_rn(0.f);
            #pragma unroll 2
            for (int v = tid; v < nv; v += kConsumers) hm = absmax8(x_s[v], hm);
            float mx = fmaxf(__low2float(hm), __high2float(hm));
            mx = warp_max(mx);
            if (lane == 0) max_s[warp] = mx;
        } else {
            #pragma unroll
            for (int m = 0; m < MT; ++m) {
                __half2 hm = __float2half2_rn(0.f);
                if (m < M) {
                    const uint4* xv = reinterpret_cast<const uint4*>(a.X + (int64_t)m * K);
                    #pragma unroll 4
                    for (int v = tid; v < nv; v += kConsumers) hm = absmax8(xv[v], hm);
                }
                float mx = fmaxf(__low2float(hm), __high2float(hm));
                mx = warp_max(mx);
                if (lane == 0) max_s[warp * MT + m] = mx;
            }
        }
        named_bar_sync(1, kConsumers);
        #pragma unroll
        for (int m = 0; m < MT; ++m) {
            float mx = 0.f;
            #pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) mx = fmaxf(mx, max_s[w * MT + m]);
            sa_r[m] = __fdiv_rn(mx, 127.f);
            const float rs = sa_r[m] > 0.f ? __frcp_rn(sa_r[m]) : 0.f;
            const float r_lo = __fmul_rn(rs, 1.f - 0x1p-21f);
            const float r_hi = __fmul_rn(rs, 1.f + 0x1p-21f);
            if (m < M) {
                if (staged)
                    quant_piece(x_s + v0, act_w, sa_r[m], r_lo, r_hi);
                else
                    quant_piece(reinterpret_cast<const uint4*>(a.X + (int64_t)m * K) + v0,
                                act_w + m * act_words, sa_r[m], r_lo, r_hi);
            }
        }
        named_bar_sync(1, kConsumers);
        if (a.Xq_out != nullptr && rb == 0) {
            for (int m = 0; m < M; ++m) {
                const uint32_t* src = act_w + m * act_words;
                for (int v = tid; v < nvq; v += kConsumers) {
                    const uint32_t e = src[v], o = src[plane + v];
                    *reinterpret_cast<uint2*>(a.Xq_out + (int64_t)m * K + 8 * (int64_t)(v0 + v)) =
                        make_uint2(__byte_perm(e, o, 0x5140), __byte_perm(e, o, 0x7362));
                }
            }
        }
        if (a.sa_out != nullptr && blockIdx.x == 0) {
            #pragma unroll
            for (int m = 0; m < MT; ++m)
                if (tid == m && m < M) a.sa_out[m] = sa_r[m];
        }
        #pragma unroll
        for (int m = 0; m < MT; ++m) {
            #pragma unroll
            for (int s = 0; s < SMAX; ++s) {
                const int c = j + s * Cl;
                if (m < M && s < ncol) {
                    const uint4* src = reinterpret_cast<const uint4*>(act_w + m * act_words);
                    const uint4 e = src[c], o = src[pl.Gq + c];
                    act[m][s][0] = e.x; act[m][s][1] = e.y; act[m][s][2] = e.z; act[m][s][3] = e.w;
                    act[m][s][4] = o.x; act[m][s][5] = o.y; act[m][s][6] = o.z; act[m][s][7] = o.w;
                } else {
                    #pragma unroll
                    for (int t = 0; t < kActWords; ++t) act[m][s][t] = 0u;
                }
            }
        }
    } else {
        if constexpr (!kW4) {
            // W8: this piece of every activation row, copied once per CTA
            if (pl.x_bytes > 0) {
                uint4* x_s = reinterpret_cast<uint4*>(smem + pl.off_x);
                const int nvp = gp * 2;  // 16-byte vectors per row piece
                for (int v = tid; v < M * nvp; v += kConsumers) {
                    const int m = v / nvp, u = v - m * nvp;
                    cp_async_16(smem_u32(x_s + v), a.X + (int64_t)m * K + (int64_t)g0 * 16 + 8 * u);
                }
                cp_async_wait_all();
                named_bar_sync(1, kConsumers);
            }
        }
        #pragma unroll
        for (int m = 0; m < MT; ++m) {
            if constexpr (kW4) sa_r[m] = (m < M) ? a.sa[m] : 0.f;
            #pragma unroll
            for (int s = 0; s < SMAX; ++s) {
                const int c = j + s * Cl;
                if (m < M && s < ncol) {
                    if constexpr (kW4) {
                        const int8_t* src = a.Xq + (int64_t)m * K + (int64_t)(g0 + c) * 32;
                        permute_act(ld_global_nc_v4(src), ld_global_nc_v4(src + 16), act[m][s]);
                    } else {
                        // the 16 binary16 values of the granule, kept as pairs
                        // (from the staged piece when there is one)
                        const uint4* src = pl.x_bytes > 0
                            ? reinterpret_cast<const uint4*>(smem + pl.off_x) + (m * gp + c) * 2
                            : reinterpret_cast<const uint4*>(a.X + (int64_t)m * K + (int64_t)(g0 + c) * 16);
                        const uint4 h0 = src[0];
                        const uint4 h1 = src[1];
                        act[m][s][0] = h0.x; act[m][s][1] = h0.y; act[m][s][2] = h0.z; act[m][s][3] = h0.w;
                        act[m][s][4] = h1.x; act[m][s][5] = h1.y; act[m][s][6] = h1.z; act[m][s][7] = h1.w;
                    }
                } else {
                    #pragma unroll
                    for (int t = 0; t < kActWords; ++t) act[m][s][t] = 0u;
                }
            }
        }
    }


    // W4: the low nibbles enter the dot product biased by +8 (n ^ 8 = q + 8),
    // so each row's sum carries 8 * (sum of the even-k codes) too much.
    int corr[MT];
    #pragma unroll
    for (int m = 0; m < MT; ++m) {
        corr[m] = 0;
        if constexpr (kW4) {
            #pragma unroll
            for (int s = 0; s < SMAX; ++s)
                #pragma unroll
                for (int t = 0; t < 4; ++t) corr[m] = __dp4a((int)act[m][s][t], 0x08080808, corr[m]);
        }
    }
    // the weight-scale cache must have landed before any output is written
    wait_or_abort(smem_u32(sw_bar), 0, abort_flag, kErrFullWait);

    // ------------------------------------------------------ streaming loop
    // Stages are consumed in batches of kBatch: per stage each thread only
    // multiplies and accumulates; the cross-thread reduction and the outputs
    // of a whole batch follow together, so their latencies overlap.
    constexpr int kBatch = 2;
    constexpr int NCH = MT == 1 ? 2 : 1;       // independent chains per sum
    AccT* red = reinterpret_cast<AccT*>(smem + pl.off_red);  // [2][warps][kBatch][MT]
    const int wpr = Cl >> 5;                                  // warps per row-piece
    // Every thread loads SMAX granules per row-piece; columns past this
    // thread's last valid one are clamped to a valid address and multiply
    // zero activations, so the loads need no branch and can all be issued
    // before the arithmetic.
    int coff[SMAX];
    #pragma unroll
    for (int s = 0; s < SMAX; ++s)
        coff[s] = i * RBp + min(j + s * Cl, gp - 1) * kGranBytes;
    int slot = 0;
    uint32_t fph = 0;  // parity of the full phase being waited for
    for (int sb = 0; sb < nstages; sb += kBatch) {
        AccT part[kBatch][MT];
        #pragma unroll
        for (int d = 0; d < kBatch; ++d) {
            #pragma unroll
            for (int m = 0; m < MT; ++m) part[d][m] = 0;
            if (sb + d < nstages) {  // uniform over the CTA
                wait_or_abort(smem_u32(full + slot), fph, abort_flag, kErrFullWait);
                const uint8_t* stage = smem + slot * pl.stage_stride;
                uint4 wg[SMAX];
                #pragma unroll
                for (int s = 0; s < SMAX; ++s)
                    wg[s] = *reinterpret_cast<const uint4*>(stage + coff[s]);
                __syncwarp();
                if (lane == 0) {
                    // the last warp done with this slot refills it with the
                    // stage NS further on
                    __threadfence_block();
                    if (atomicAdd(released + slot, 1) == kConsumerWarps - 1) {
                        released[slot] = 0;
                        __threadfence_block();
                        if (sb + d + NS < nstages && !*abort_flag) issue(sb + d + NS, slot);
                    }
                }
                if (++slot == NS) { slot = 0; fph ^= 1u; }

                using LaneT = typename std::conditional<kW4, int, float>::type;
                LaneT alo[MT][NCH], ahi[MT][NCH];
                #pragma unroll
                for (int m = 0; m < MT; ++m) {
                    #pragma unroll
                    for (int h = 0; h < NCH; ++h) { alo[m][h] = 0; ahi[m][h] = 0; }
                }
                #pragma unroll
                for (int s = 0; s < SMAX; ++s) {
                    if (kExactS || s < pl.S) {  // uniform over the CTA
                        const uint32_t wv[4] = {wg[s].x, wg[s].y, wg[s].z, wg[s].w};
                        #pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            if constexpr (kW4) {
                                // low nibbles: (n ^ 8) = q + 8 in [0, 15]; high
                                // nibbles left in place read as int8 = 16 * q
                                const uint32_t lo = (wv[t] ^ 0x08080808u) & 0x0F0F0F0Fu;
                                const uint32_t hi = wv[t] & 0xF0F0F0F0u;
                                #pragma unroll
                                for (int m = 0; m < MT; ++m) {
                                    LaneT& cl = alo[m][t % NCH];
                                    LaneT& ch = ahi[m][t % NCH];
                                    cl = __dp4a((int)lo, (int)act[m][s][t], cl);
                                    ch = __dp4a((int)hi, (int)act[m][s][4 + t], ch);
                                }
                            } else {
                                // int8 code q -> binary16 exactly: the byte uu = q + 128
                                // under the high byte 0x64 encodes 1024 + q + 128; one
                                // packed subtraction of 1152 leaves q (|q| <= 128)
                                const uint32_t u = wv[t] ^ 0x80808080u;
                                const uint32_t p01 = __byte_perm(u, 0x64646464u, 0x4140);
                                const uint32_t p23 = __byte_perm(u, 0x64646464u, 0x4342);
                                const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6480));
                                const __half2 h01 = __hsub2(*reinterpret_cast<const __half2*>(&p01), bias);
                                const __half2 h23 = __hsub2(*reinterpret_cast<const __half2*>(&p23), bias);
                                const uint32_t q01 = *reinterpret_cast<const uint32_t*>(&h01);
                                const uint32_t q23 = *reinterpret_cast<const uint32_t*>(&h23);
                                #pragma unroll
                                for (int m = 0; m < MT; ++m) {
                                    LaneT& c0 = alo[m][t % NCH];
                                    LaneT& c1 = ahi[m][t % NCH];
                                    fma_f16_f32x2(c0, c1, q01, act[m][s][2 * t]);      // codes 4t, 4t+1
                                    fma_f16_f32x2(c0, c1, q23, act[m][s][2 * t + 1]);  // codes 4t+2, 4t+3
                                }
                            }
                        }
                    }
                }
                #pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if constexpr (kW4) {
                        int lo_sum = 0, hi_sum = 0;
                        #pragma unroll
                        for (int h = 0; h < NCH; ++h) { lo_sum += alo[m][h]; hi_sum += ahi[m][h]; }
                        part[d][m] = lo_sum - corr[m] + (hi_sum >> 4);  // exact: hi_sum = 16 * sum
                    } else {
                        float sum = 0.f;
                        #pragma unroll
                        for (int h = 0; h < NCH; ++h) sum += alo[m][h] + ahi[m][h];
                        part[d][m] = sum;
                    }
                }
            }
        }

        // reduce the batch across the Cl threads of each row-piece
        #pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            if (o < Cl) {
                #pragma unroll
                for (int d = 0; d < kBatch; ++d)
                    #pragma unroll
                    for (int m = 0; m < MT; ++m)
                        part[d][m] += __shfl_xor_sync(0xFFFFFFFFu, part[d][m], o);
            }
        }
        if (wpr > 1) {
            AccT* rbuf = red + ((sb / kBatch) & 1) * kConsumerWarps * kBatch * MT;
            if (lane == 0) {
                #pragma unroll
                for (int d = 0; d < kBatch; ++d)
                    #pragma unroll
                    for (int m = 0; m < MT; ++m) rbuf[(warp * kBatch + d) * MT + m] = part[d][m];
            }
            // only the wpr warps of this row-piece meet (barrier 2 + i; at
            // most 4 row-pieces when a row-piece spans warps)
            named_bar_sync(2 + i, Cl);
            if (j == 0) {
                #pragma unroll
                for (int d = 0; d < kBatch; ++d)
                    #pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        AccT t = rbuf[(warp * kBatch + d) * MT + m];
                        for (int w = 1; w < wpr; ++w) t += rbuf[((warp + w) * kBatch + d) * MT + m];
                        part[d][m] = t;
                    }
            }
        }
        if (j == 0) {
            #pragma unroll
            for (int d = 0; d < kBatch; ++d) {
                const int r = (sb + d) * pl.Rl + i;   // row within this CTA's range
                if (sb + d < nstages && r < nrows) {
                    const int64_t n = row0 + r;
                    if (pl.P == 1) {
                        const float swv = kW4 ? sw_s[r]
                                              : __half2float(reinterpret_cast<const __half*>(sw_s)[r + (row0 & 1)]);
                        const int sg = segment_of(a, n);
                        const int64_t Ng = a.off[sg + 1] - a.off[sg];
                        float* Yp = a.Yg[sg] + (n - a.off[sg]);
                        #pragma unroll
                        for (int m = 0; m < MT; ++m) {
                            if (m < M) {
                                if constexpr (kW4) {
                                    Yp[m * Ng] = __fmul_rn(__fmul_rn(__int2float_rn(part[d][m]), swv), sa_r[m]);
                                    if (a.acc_out != nullptr) a.acc_out[m * N + n] = part[d][m];
                                } else {
                                    Yp[m * Ng] = __fmul_rn(part[d][m], swv);
                                }
                            }
                        }
                    } else {
                        AccT* pbuf = static_cast<AccT*>(a.part);
                        #pragma unroll
                        for (int m = 0; m < MT; ++m)
                            if (m < M) pbuf[((int64_t)p * M + m) * N + n] = part[d][m];
                    }
                }
            }
        }
    }

    // After an abandoned wait, copies may still be landing: wait for them
    // (bounded) so that none writes shared memory after the CTA exits.
    if (*abort_flag && tid == 0) {
        for (int s2 = (nstages > NS ? nstages - NS : 0); s2 < nstages; ++s2)
            if (!mbar_wait(smem_u32(full + s2 % NS), (s2 / NS) & 1))
                atomicOr(&g_device_error, kErrDrainWait);
    }
    if (pl.P == 1) {
        if (a.H != nullptr) {
            // the CTA's outputs were written by its own threads: a barrier makes
            // them visible, then each pair of rows gives one gated product
            named_bar_sync(1, kConsumers);
            if (!*abort_flag) silu_pairs(a, row0, nrows, tid);
        }
        return;
    }

    // ---------------------------------------------- split-K: last CTA sums
    __threadfence();
    named_bar_sync(1, kConsumers);
    if (tid == 0) *last_flag = (atomicAdd(a.tickets + rb, 1u) == (unsigned)(pl.P - 1));
    named_bar_sync(1, kConsumers);
    if (!*last_flag) return;
    __threadfence();
    const AccT* part = static_cast<const AccT*>(a.part);
    for (int r = tid; r < nrows; r += kConsumers) {
        const int64_t n = row0 + r;
        const int sg = segment_of(a, n);
        const int64_t ng = n - a.off[sg];
        const int64_t Ng = a.off[sg + 1] - a.off[sg];
        float swv = 0.f;
        if constexpr (kW4)
            swv = static_cast<const float*>(a.wscale[sg])[ng];
        else
            swv = __half2float(static_cast<const __half*>(a.wscale[sg])[ng]);
        #pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < M) {
                AccT t = 0;
                for (int q = 0; q < pl.P; ++q) t += __ldcg(part + ((int64_t)q * M + m) * N + n);
                if constexpr (kW4) {
                    a.Yg[sg][m * Ng + ng] = __fmul_rn(__fmul_rn(__int2float_rn(t), swv), sa_r[m]);
                    if (a.acc_out != nullptr) a.acc_out[m * N + n] = t;
                } else {
                    a.Yg[sg][m * Ng + ng] = __fmul_rn(t, swv);
                }
            }
        }
    }
    if (a.H != nullptr) {
        named_bar_sync(1, kConsumers);
        silu_pairs(a, row0, nrows, tid);
    }
    if (tid == 0) a.tickets[rb] = 0u;  // ready for the next call
}

// --------------------------------------------------------------- launching

template <bool kW4, int MT, int SMAX, bool kFused, bool kExactS = false>
static cudaError_t launch_one(const GemvArgs& args, unsigned flags, cudaStream_t stream) {
    auto* fn = gemv_kernel<kW4, MT, SMAX, kFused, kExactS>;
    static int attr_set[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_set[dev]) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
        if (e != cudaSuccess) return e;
        // Carve out all of L1 as shared memory so a CTA of the next kernel
        // (programmatic dependent launch) fits beside the running one.
        e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        attr_set[dev] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(args.pl.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = args.pl.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (flags & 1u) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, fn, args);
}

static void set_segments(GemvArgs& a, int G, const uint8_t* const* W, const void* const* s,
                         const int64_t* Ns, float* const* Y) {
    int64_t off = 0;
    for (int k = 0; k < kMaxSegments; ++k) {
        a.off[k] = off;
        if (k < G) {
            a.W[k] = W[k];
            a.wscale[k] = s[k];
            a.Yg[k] = Y[k];
            off += Ns[k];
        }
    }
    a.off[kMaxSegments] = off;
    for (int k = G; k < kMaxSegments; ++k) a.off[k] = off;  // empty tail segments
}

}  // namespace w4a8
