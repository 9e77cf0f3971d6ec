// rowdot_plan.h -- launch plan of the row-per-thread dp4a kernels
// (rowdot.cu): W4A8 with row-wise scales for 2..8 activation rows, and with
// group-wise scales for 1..8 (one thread per weight row).
#pragma once

#include <cstddef>

namespace w4a8 {

// Launch plan of the row-per-thread dp4a kernel (csrc/rowdot.cu).
constexpr int kRowdotMaxM = 8;        // batch rows the kernel is instantiated for: 2..8
constexpr int kRowdotDefaultTPR = 4;  // threads per weight row (one CTA of 512 per SM)
struct RowdotPlan {
    int MT;            // activation rows (2..kRowdotMaxM)
    int tpr, cps;      // threads per weight row, CTAs per SM
    int tiles;         // 128-row weight tiles
    int nbox;          // 256-code K boxes (K rounded up)
    int P, bpp;        // K pieces, boxes per piece
    int NS;            // weight ring slots of 16 KB
    int gshift;        // group scales: groups of 2^gshift codes (-1: row-wise)
    int lshift, nch;   // group scales: chunks of 2^lshift codes, nch of them
    int force_p;       // group scales: requested K pieces (0 = by the tiles)
    int cps_req;       // group scales: requested CTAs per SM (0 = by the grid)
    int nph, abox;     // group scales: thread phases per CTA (= tpr), boxes per chunk
    int grid, smem, sms;
    size_t off_sa, off_codes, off_part;  // workspace layout
    size_t ws_bytes;
};

}  // namespace w4a8
