// plan.h -- launch plan of the streaming GEMV kernels (host and device).
//
// A weight row is cut into 16-byte granules (32 INT4 codes, or 16 INT8
// codes).  The K dimension may be split into P pieces ("split-K"); each CTA
// streams a contiguous range of rows of one piece through a shared-memory
// ring.  Inside a stage, `Cl` consumer threads share one row-piece: thread j
// owns granule columns j, j+Cl, j+2Cl, ... (at most S of them), so the
// activation values it multiplies never change and stay in registers.
#pragma once

#include <cstddef>
#include <cstdint>

namespace w4a8 {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;  // 256 consumer threads
constexpr int kThreads = kConsumers;             // thread 0 also issues the copies
constexpr int kGranBytes = 16;
constexpr int kMaxSplits = 16;
constexpr int kMaxRowsPerCta = 4096;              // bounds the scale cache in smem
constexpr int kMaxSmem = 232448;                  // 227 KB opt-in limit per CTA
constexpr int kMaxSmem2 = 233472 / 2 - 1024;      // per CTA with two CTAs on an SM
// A single fp16 activation row up to this size is staged in shared memory
// (fused W4A8, M == 1).
constexpr int kMaxXStage = 40960;
constexpr int kDefaultRingBytes = 96 * 1024;
// Split-K workspace layout: arrival counters first, at a fixed place, so any
// call leaves them zero for the next call whatever its shape; partials after.
constexpr int kTicketSlots = 1024;
constexpr size_t kTicketBytes = kTicketSlots * 4;

struct GemvPlan {
    int MT;            // activation rows rounded up to 1, 2, 4 or 8
    int smax;          // compile-time bound on granule columns per thread
    int P;             // K pieces
    int Gt;            // granules per full weight row
    int Gq;            // granules per piece (the last piece may have fewer)
    int Cl, log2Cl;    // threads per row-piece
    int S;             // granule columns per thread
    int Rl;            // row-pieces per stage (kConsumers / Cl)
    int Gs;            // CTAs per piece
    int grid;          // Gs * P
    int rows_max;      // most rows any CTA streams
    int NS;            // ring stages
    int stage_stride;  // bytes per ring stage (multiple of 128)
    int cps;           // CTAs per SM the grid was sized for
    int x_bytes;       // staged activation row (0: read from global memory)
    int off_bars, off_sw, off_x, off_act, off_red, off_max, off_flag;
    int smem;          // dynamic shared memory bytes
    size_t ws_bytes;   // workspace: kTicketBytes of counters + [P][M][N] x 4
                       // bytes of partials; 0 when P == 1
};

struct Tuning {
    int force_splits;   // 0 = heuristic, else P
    int force_cl;       // 0 = heuristic, else threads per row-piece
    int ring_bytes;     // 0 = default ring size
    int ctas_per_sm;    // 0 = default (1), else CTAs per SM per K piece
};

// Launch plan of the tensor-core path (csrc/mma.cu).
struct MmaPlan {
    int BN;            // batch rows padded to a multiple of 16 (the MMA's N)
    int tiles;         // 128-row weight tiles
    int nkb;           // 64-wide K blocks
    int P, kbp;        // K pieces, K blocks per piece
    int force_p;       // requested K pieces (0 = by the tiles)
    int grid, smem, sms;
    int stages, stage_bytes;             // weight ring
    size_t off_sa, off_sum, off_codes, off_part, off_acc;  // workspace layout
    size_t ws_bytes;
};

inline int round_up(int v, int a) { return (v + a - 1) / a * a; }
inline size_t round_up_sz(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline int mt_of(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8; }

// Builds the plan; returns false when no valid plan exists for the shape.
// w4: INT4 weights (32 codes per granule) else INT8 (16 per granule).
// pair: the rows come in pairs (the gated product of gate/up rows 2i, 2i+1)
// and every CTA takes whole pairs.
inline bool make_gemv_plan(bool w4, bool fused, int M, int64_t K, int64_t N, int num_sms,
                           const Tuning& tu, GemvPlan* out,
                           bool pair = false) {
    if (pair && (N < 2 || N % 2)) return false;
    GemvPlan pl = {};
    pl.MT = mt_of(M);
    pl.smax = 8 / pl.MT;  // 8 activation registers per granule and row (W4 codes, W8 binary16 pairs)
    if (pl.smax < 1) return false;
    const int kgran = w4 ? 32 : 16;
    if (K % kgran) return false;
    pl.Gt = (int)(K / kgran);
    double best_cost = 1e300;
    bool found = false;
    for (int P = 1; P <= kMaxSplits; ++P) {
        if (tu.force_splits && P != tu.force_splits) continue;
        const int Gq = (pl.Gt + P - 1) / P;
        if ((P - 1) * Gq >= pl.Gt) continue;  // last piece must be non-empty
        int bestCl = -1, bestS = 0;
        double bestU = 0.0;
        for (int lc = 0; lc <= 8; ++lc) {
            const int Cl = 1 << lc;
            if (tu.force_cl && Cl != tu.force_cl) continue;
            const int S = (Gq + Cl - 1) / Cl;
            if (S > pl.smax) continue;
            const double u = (double)Gq / ((double)Cl * S);
            if (u > bestU + 1e-9) { bestU = u; bestCl = Cl; bestS = S; }
        }
        if (bestCl < 0) continue;
        // Two CTAs per SM double the consumer warps that hide the per-stage
        // latency; keep one when a CTA would get fewer than two stages.
        int cps = tu.ctas_per_sm;
        if (cps <= 0) {
            const int64_t gs2 = (int64_t)num_sms * 2 / P;
            const int rl = kConsumers / bestCl;
            cps = (gs2 >= 1 && N / gs2 >= 2 * rl) ? 2 : 1;
        }
        int64_t Gs = (int64_t)num_sms * cps / P;
        if (Gs < 1) Gs = 1;
        if (Gs > (pair ? N / 2 : N)) Gs = pair ? N / 2 : N;
        if (P > 1 && Gs > kTicketSlots) Gs = kTicketSlots;
        auto rows_of = [&](int64_t gs) { return pair ? 2 * ((N / 2 + gs - 1) / gs) : (N + gs - 1) / gs; };
        int64_t rows_max = rows_of(Gs);
        while (P == 1 && rows_max > kMaxRowsPerCta) {  // keep the scale cache small
            Gs += (int64_t)num_sms * cps;
            rows_max = rows_of(Gs);
        }
        if (Gs * P > 0x7FFFFFFF) continue;
        // Streaming cost ~ granules per CTA; low lane utilisation only costs
        // when the integer pipe becomes the limit (larger M); a split pays a
        // partial-sum pass and an extra serial step at the end.
        double cost = (double)rows_max * Gq * cps / 2.0;  // per-SM share of the stream
        const double alu = 0.3 * pl.MT / bestU;
        if (alu > 1.0) cost *= alu;
        if (P > 1) cost = cost * 1.05 + 2800.0;
        if (cost < best_cost) {
            best_cost = cost;
            found = true;
            pl.cps = cps;
            pl.P = P;
            pl.Gq = Gq;
            pl.Cl = bestCl;
            pl.S = bestS;
            pl.Gs = (int)Gs;
            pl.rows_max = (int)rows_max;
        }
    }
    if (!found) return false;
    pl.log2Cl = 0;
    while ((1 << pl.log2Cl) < pl.Cl) ++pl.log2Cl;
    pl.Rl = kConsumers / pl.Cl;
    pl.grid = pl.Gs * pl.P;

    const int stage_bytes = pl.Rl * pl.Gq * kGranBytes;
    pl.stage_stride = round_up(stage_bytes, 128);
    const int ring = tu.ring_bytes > 0 ? tu.ring_bytes : kDefaultRingBytes;
    int NS = ring / pl.stage_stride;
    if (NS < 2) NS = 2;
    if (NS > 16) NS = 16;

    const int sw_bytes = pl.P == 1 ? round_up(pl.rows_max * 4 + 8, 16) : 0;
    const int act_bytes = (w4 && fused) ? round_up(pl.MT * pl.Gq * 32, 128) : 0;
    // the K piece of the activation rows a W8 CTA reads, staged once per CTA
    const int w8_x = w4 ? 0 : M * pl.Gq * kGranBytes * 2;
    pl.x_bytes = (w4 && fused && pl.MT == 1 && 2 * K <= kMaxXStage) ? (int)(2 * K)
               : (!w4 && w8_x <= kMaxXStage) ? w8_x : 0;
    const int red_bytes = 2 * kConsumerWarps * 4 * pl.MT * 4;  // [2][warps][batch 4][MT]
    const int max_bytes = kConsumerWarps * pl.MT * 4;
    // Shrink the ring until the CTA fits beside its sibling(s) on an SM; if
    // even two stages do not fit, fall back to the one-CTA limit.
    const int limit = (pl.cps >= 2) ? kMaxSmem2 : kMaxSmem;
    for (;; --NS) {
        int off = NS * pl.stage_stride;
        pl.off_bars = off;
        off += NS * 8 + 8 + NS * 4;  // full[NS], scale-cache mbarrier, released[NS]
        pl.off_sw = round_up(off, 16);
        off = pl.off_sw + sw_bytes;
        pl.off_x = round_up(off, 128);
        off = pl.off_x + pl.x_bytes;
        pl.off_act = round_up(off, 128);
        off = pl.off_act + act_bytes;
        pl.off_red = round_up(off, 16);
        off = pl.off_red + red_bytes;
        pl.off_max = off;
        off += max_bytes;
        pl.off_flag = round_up(off, 16);
        off = pl.off_flag + 16;
        pl.smem = round_up(off, 128);
        if (pl.smem <= limit || (NS <= 2 && pl.smem <= kMaxSmem)) break;
        if (NS <= 2) return false;
    }
    pl.NS = NS;
    if (pl.P > 1) pl.ws_bytes = kTicketBytes + round_up_sz((size_t)pl.P * M * N * 4, 256);
    *out = pl;
    return true;
}

}  // namespace w4a8
