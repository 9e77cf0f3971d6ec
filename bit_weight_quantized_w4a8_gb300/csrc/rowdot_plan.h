// rowdot_plan.h -- launch plan of the row-per-thread dp4a kernel
// (rowdot.cu): W4A8 with row-wise scales for 2..8 activation rows.
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
    int gwin, gstride; // groups staged per CTA, floats per staged row
    int grid, smem, sms;
    size_t off_sa, off_codes, off_part;  // workspace layout
    size_t ws_bytes;
};

}  // namespace w4a8
