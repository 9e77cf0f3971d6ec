// actq.cuh -- the dynamic per-row INT8 activation quantizer of the Jetson
// INT4 page (sections 正确方向 / 当前实现方式) for 8 binary16 values at a
// time, shared by the dp4a and tensor-core kernels.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

namespace w4a8 {

// Activation codes, clamp(round_half_away(x / s), +-127) with the IEEE
// quotient x / s, for 8 binary16 values at once, split by parity: .x holds
// the codes of elements 0, 2, 4, 6 and .y those of 1, 3, 5, 7 (low byte
// first), the order in which the packed weights present them.
//
// Exact slow form: one IEEE division and roundf per value.
static __device__ __noinline__ uint2 quant8_split_exact(uint4 h, float s) {
    if (!(s > 0.f)) return make_uint2(0u, 0u);
    const __half* p = reinterpret_cast<const __half*>(&h);
    uint32_t w[2] = {0u, 0u};
    #pragma unroll
    for (int k = 0; k < 8; ++k) {
        int q = static_cast<int>(roundf(__fdiv_rn(__half2float(p[k]), s)));
        q = min(max(q, -127), 127);
        w[k & 1] |= (uint32_t)(q & 0xFF) << (8 * (k >> 1));
    }
    return make_uint2(w[0], w[1]);
}

// Fast form, given r_lo and r_hi, rcp_rn(s) scaled by 1 -+ 2^-21 and
// rounded (both 0 when s = 0).  They bracket 1/s with a relative margin of
// more than 2^-22 on each side, so for x != 0 the IEEE quotient x / s (within
// 2^-24 relative of the exact one) lies strictly between x * r_lo and
// x * r_hi.  With M = 1.5 * 2^23, fma(x, r, M) holds rint(x * r) of the exact
// product in the low bits of its encoding (|x * r| < 2^22).  When the two
// ends round to the same integer k, both lie in [k - 1/2, k + 1/2] and the
// quotient strictly inside, so k is the code and no tie is involved; since
// |x| <= 127 * s up to one rounding of s, |k| <= 127 needs no clamp.  A
// vector in which some value's ends disagree (a half-integer between them,
// about one value in 10^4 at most) takes the exact form.
static __device__ __forceinline__ uint2 quant8_split(uint4 h, float s, float r_lo, float r_hi) {
    constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
    const __half2* p = reinterpret_cast<const __half2*>(&h);
    uint32_t y[8];
    uint32_t diff = 0u;
    #pragma unroll
    for (int t = 0; t < 4; ++t) {
        const float2 f = __half22float2(p[t]);
        const uint32_t a0 = __float_as_uint(__fmaf_rn(f.x, r_lo, kMagic));
        const uint32_t b0 = __float_as_uint(__fmaf_rn(f.x, r_hi, kMagic));
        const uint32_t a1 = __float_as_uint(__fmaf_rn(f.y, r_lo, kMagic));
        const uint32_t b1 = __float_as_uint(__fmaf_rn(f.y, r_hi, kMagic));
        diff |= (a0 ^ b0) | (a1 ^ b1);
        y[2 * t] = a0;
        y[2 * t + 1] = a1;
    }
    if (diff != 0u) return quant8_split_exact(h, s);
    // the low byte of y is k modulo 256, the code's two's complement byte
    const uint32_t ev = __byte_perm(__byte_perm(y[0], y[2], 0x0040), __byte_perm(y[4], y[6], 0x0040), 0x5410);
    const uint32_t od = __byte_perm(__byte_perm(y[1], y[3], 0x0040), __byte_perm(y[5], y[7], 0x0040), 0x5410);
    return make_uint2(ev, od);
}

// The bracket of 1/s the fast form needs (both 0 when s = 0).
__device__ __forceinline__ void quant_bracket(float s, float* r_lo, float* r_hi) {
    const float r = s > 0.f ? __frcp_rn(s) : 0.f;
    *r_lo = __fmul_rn(r, 1.f - 0x1p-21f);
    *r_hi = __fmul_rn(r, 1.f + 0x1p-21f);
}

}  // namespace w4a8
