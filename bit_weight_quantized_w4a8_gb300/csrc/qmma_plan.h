// qmma_plan.h -- launch plan of the warp-level e4m3 MMA kernel (qmma.cu):
// W4A8 with row-wise scales for 2..32 activation rows.
#pragma once

#include <cstddef>

namespace w4a8 {

constexpr int kQmmaMaxM = 32;  // batch rows the kernel is instantiated for: 2..32

struct QmmaPlan {
    int M;             // activation rows (2..kQmmaMaxM)
    int h16;           // 1: binary16 operands (m16n8k16), 0: e4m3 (m16n8k32)
    int NT;            // n-tiles of 8 MMA columns: ceil(M / 8) batch rows (binary16) or
                       // ceil(M / 4) (e4m3: 4 batch rows x {high, low} each)
    int R;             // 16-row MMA tiles per warp (= boxes interleaved over R warp groups)
    int tiles;         // 128-row weight tiles
    int nbox;          // 256-code K boxes (K rounded up)
    int P, bpp;        // K pieces, boxes per piece
    int NS;            // ring stages (weight box + activation slice)
    int stage_bytes;   // 16384 + activation slice (4096 NT binary16, 2048 NT e4m3)
    int pre_pieces;    // CTAs per batch row of the activation pass
    int persist;       // 1: one CTA per SM walks the tiles b, b + grid, ... (one K piece)
    int grid, smem, sms;
    size_t off_sa, off_sum, off_codes, off_part;  // workspace layout
    size_t ws_bytes;
};

}  // namespace w4a8
