/*
 * oracle.c -- plain, single-threaded CPU definition of the weight-quantized
 * decode linear layer (W4A8 and W8A16) and of the IndexSoftmax operator.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark do.  It shares no code, header, table or constant
 * generator with the CUDA library.
 *
 * Sources (pages that define the method):
 *  [P1] "Jetson Orin AGX 上的 INT4 量化推理实践：从 9 tok/s 到 19.6 tok/s",
 *       sections 当前实现方式 (row-wise INT4 weight with one scale per row;
 *       activation dynamically quantized to INT8 before every linear;
 *       output = int32 accumulate * weight_scale * activation_scale) and
 *       正确方向 (INT4 weight, INT8 activation, int32 accumulate, float out),
 *       and 后续优化方向 (group-wise scales, listed as the next step: read
 *       as the row-wise definition applied to each group of gs codes).
 *  [P2] "TPU-MLIR W8A16 for ChatGLM2-6B", section 2 (per-channel INT8
 *       weights) and section 4 (the five steps: load, cast INT8 to F16,
 *       multiply by the scale, matrix multiply with the activation, store).
 *  [P3] "【MLSys 2026】IntAttention：全整数注意力流水线，边缘推理的高效部署",
 *       section 基准/方法设计 (IndexSoftmax: integer clipping of the row
 *       distances, a 2^b-entry UINT8 exponent table, integer normalization
 *       to UINT8 probabilities).
 * Where the pages leave a step open, the reading used is stated at the
 * function (symmetric codes, divisors 7 and 127, round half away from zero,
 * true division, low-nibble-first two's-complement packing, fp32 rescale in
 * the order (acc * s_w) * s_a; for group scales a binary64 reference plus
 * the magnitude that bounds any fp32 evaluation of it, and the binary32
 * evaluation in the library's fixed order: exact group sums folded with one
 * fused multiply-add each inside chunks of max(gs, 1024) codes, chunk
 * results added in ascending order).
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared (no fast-math, no
 * FMA contraction, so every float operation is one IEEE binary32 operation).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_SHAPE 3
#define ORACLE_ERR_OVERFLOW 6

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 <-> binary32, written from the format's definition.      */
/* ------------------------------------------------------------------------ */

/* binary16 bits -> float (always exact). */
float oracle_half_to_float(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    float v;
    if (e == 0x1F) {
        v = m ? NAN : INFINITY;
    } else if (e == 0) {
        v = ldexpf((float)m, -24);          /* subnormal: m * 2^-24 */
    } else {
        v = ldexpf((float)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* float -> binary16 bits, round to nearest, ties to even. */
uint16_t oracle_float_to_half(float f)
{
    uint32_t x;
    memcpy(&x, &f, 4);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    uint32_t ax = x & 0x7FFFFFFFu;
    if (ax > 0x7F800000u) return (uint16_t)(sign | 0x7E00u);   /* NaN */
    if (ax == 0x7F800000u) return (uint16_t)(sign | 0x7C00u);  /* inf */
    if (ax < 0x00800000u) return sign;  /* float subnormal: far below 2^-25 */

    int e = (int)(ax >> 23) - 127;               /* |f| = m24 * 2^(e-23) */
    uint32_t m24 = (ax & 0x7FFFFFu) | 0x800000u;
    int eh = e < -14 ? -14 : e;                  /* binary16 exponent used */
    /* quantum of the result is 2^(eh-10); n = |f| / quantum = m24 >> shift */
    int shift = 13 + eh - e;
    uint32_t n;
    if (shift >= 32) {
        n = 0;
    } else {
        n = m24 >> shift;
        uint32_t rem = m24 & ((1u << shift) - 1u);
        uint32_t half = 1u << (shift - 1);
        if (rem > half || (rem == half && (n & 1u))) n += 1;
    }
    /* eh == -14: n is the full encoding (subnormal, or 0x400 = 2^-14).
       otherwise n in [1024, 2048]; a carry to 2048 moves to the next
       exponent naturally. */
    uint32_t bits = (eh == -14) ? n : ((uint32_t)(eh + 15) << 10) + (n - 1024u);
    if (bits >= 0x7C00u) bits = 0x7C00u;         /* overflow -> inf */
    return (uint16_t)(sign | bits);
}

/* ------------------------------------------------------------------------ */
/* Symmetric rounding quantizer shared by the definitions below.             */
/* ------------------------------------------------------------------------ */

/* q = clamp(round_half_away(v / s), -qmax, qmax); s == 0 gives 0.
   [P1 当前实现方式] weight_float ~ int4_value * weight_scale; the divisor,
   rounding and clamp are the reading stated in the file header. */
static int quant_code(float v, float s, int qmax)
{
    if (s == 0.0f) return 0;
    float t = v / s;             /* one IEEE division */
    float r = roundf(t);         /* halves go away from zero */
    if (r > (float)qmax) r = (float)qmax;
    if (r < (float)-qmax) r = (float)-qmax;
    return (int)r;
}

static float row_absmax(const float* row, int64_t K)
{
    float m = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
        float a = fabsf(row[k]);
        if (a > m) m = a;
    }
    return m;
}

/* ------------------------------------------------------------------------ */
/* a1: row-wise INT4 weight quantizer + packing  [P1 当前实现方式]            */
/* ------------------------------------------------------------------------ */

/* W[N][K] fp32 -> Wq[N][K/2] packed nibbles + sw[N] fp32.
   Per output row n: s = max|W[n,:]| / 7, q = clamp(round(W/s), -7, 7).
   Byte j of a row holds q[2j] in bits 0..3 and q[2j+1] in bits 4..7,
   each as a 4-bit two's-complement code. */
int oracle_w4_quantize(const float* W, int64_t N, int64_t K, uint8_t* Wq, float* sw)
{
    if (N < 0 || K < 0 || (K & 1)) return ORACLE_ERR_SHAPE;
    for (int64_t n = 0; n < N; ++n) {
        const float* row = W + n * K;
        float s = row_absmax(row, K) / 7.0f;
        sw[n] = s;
        for (int64_t j = 0; j < K / 2; ++j) {
            int q0 = quant_code(row[2 * j], s, 7);
            int q1 = quant_code(row[2 * j + 1], s, 7);
            Wq[n * (K / 2) + j] = (uint8_t)((q0 & 0xF) | ((q1 & 0xF) << 4));
        }
    }
    return ORACLE_OK;
}

/* Decode one 4-bit two's-complement code. */
static int nibble_value(unsigned v)
{
    return v >= 8 ? (int)v - 16 : (int)v;
}

/* Wq[N][K/2] -> q[N][K] int8 codes (inverse of the packing above). */
int oracle_w4_unpack(const uint8_t* Wq, int64_t N, int64_t K, int8_t* q)
{
    if (N < 0 || K < 0 || (K & 1)) return ORACLE_ERR_SHAPE;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t j = 0; j < K / 2; ++j) {
            uint8_t b = Wq[n * (K / 2) + j];
            q[n * K + 2 * j] = (int8_t)nibble_value(b & 0xFu);
            q[n * K + 2 * j + 1] = (int8_t)nibble_value(b >> 4);
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* a2: dynamic per-row INT8 activation quantizer  [P1 正确方向, 当前实现方式] */
/* ------------------------------------------------------------------------ */

/* X[M][K] binary16 -> Xq[M][K] int8 + sa[M] fp32.
   Per activation row m: s_a = max|x| / 127, q = clamp(round(x/s_a), -127, 127). */
int oracle_act_quantize(const uint16_t* X, int64_t M, int64_t K, int8_t* Xq, float* sa)
{
    if (M < 0 || K < 0) return ORACLE_ERR_SHAPE;
    for (int64_t m = 0; m < M; ++m) {
        float mx = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float a = fabsf(oracle_half_to_float(X[m * K + k]));
            if (a > mx) mx = a;
        }
        float s = mx / 127.0f;
        sa[m] = s;
        for (int64_t k = 0; k < K; ++k)
            Xq[m * K + k] = (int8_t)quant_code(oracle_half_to_float(X[m * K + k]), s, 127);
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* a3+a4: integer dot products  [P1 正确方向: int8 x int8 -> int32]           */
/* ------------------------------------------------------------------------ */

/* acc[m][n] = sum_k Xq[m][k] * qw[n][k], summed in int64 and checked to fit
   the int32 accumulator the pages name. */
int oracle_w4a8_dot(const int8_t* Xq, int64_t M, int64_t K, const uint8_t* Wq, int64_t N,
                    int32_t* acc)
{
    if (M < 0 || N < 0 || K < 0 || (K & 1)) return ORACLE_ERR_SHAPE;
    int status = ORACLE_OK;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            int64_t s = 0;
            for (int64_t j = 0; j < K / 2; ++j) {
                uint8_t b = Wq[n * (K / 2) + j];
                s += (int64_t)Xq[m * K + 2 * j] * nibble_value(b & 0xFu);
                s += (int64_t)Xq[m * K + 2 * j + 1] * nibble_value(b >> 4);
            }
            if (s > INT32_MAX || s < INT32_MIN) status = ORACLE_ERR_OVERFLOW;
            acc[m * N + n] = (int32_t)s;
        }
    }
    return status;
}

/* ------------------------------------------------------------------------ */
/* a5: rescale  [P1 当前实现方式: output = acc * weight_scale * act_scale]    */
/* ------------------------------------------------------------------------ */

/* Y[m][n] = ((float)acc * sw[n]) * sa[m]; two fp32 round-to-nearest
   multiplies in this order. */
void oracle_w4a8_rescale(const int32_t* acc, const float* sw, const float* sa, int64_t M,
                         int64_t N, float* Y)
{
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            float t = (float)acc[m * N + n] * sw[n];
            Y[m * N + n] = t * sa[m];
        }
    }
}

/* a-f: the whole W4A8 linear as the pages describe it: quantize the
   activation, integer dot, rescale.  Xq_out / sa_out / acc_out receive the
   intermediates (all required here; the oracle is for checking). */
int oracle_w4a8_linear(const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq,
                       const float* sw, int64_t N, float* Y, int8_t* Xq_out, float* sa_out,
                       int32_t* acc_out)
{
    int st = oracle_act_quantize(X, M, K, Xq_out, sa_out);
    if (st != ORACLE_OK) return st;
    st = oracle_w4a8_dot(Xq_out, M, K, Wq, N, acc_out);
    oracle_w4a8_rescale(acc_out, sw, sa_out, M, N, Y);
    return st;
}

/* ------------------------------------------------------------------------ */
/* b1: per-output-channel INT8 weight quantizer  [P2 sections 2 and 3]       */
/* ------------------------------------------------------------------------ */

/* W[N][K] fp32 -> Wq8[N][K] int8 + sw16[N] binary16.
   Per output channel n: s = fp16(max|W[n,:]| / 127); the codes are taken
   with that rounded scale: q = clamp(round(W / float(s)), -127, 127). */
int oracle_w8_quantize(const float* W, int64_t N, int64_t K, int8_t* Wq8, uint16_t* sw16)
{
    if (N < 0 || K < 0) return ORACLE_ERR_SHAPE;
    for (int64_t n = 0; n < N; ++n) {
        const float* row = W + n * K;
        uint16_t h = oracle_float_to_half(row_absmax(row, K) / 127.0f);
        float s = oracle_half_to_float(h);
        sw16[n] = h;
        for (int64_t k = 0; k < K; ++k) Wq8[n * K + k] = (int8_t)quant_code(row[k], s, 127);
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* b2: W8A16 product, fp64 reference  [P2 section 4, steps 2-4]              */
/* ------------------------------------------------------------------------ */

/* Y[m][n] = sum_k (q[n][k] * s[n]) * x[m][k], every product and sum in
   binary64: step 2 casts the code, step 3 multiplies by the scale
   (dequantize), step 4 multiplies with the activation. */
void oracle_w8a16_ref(const uint16_t* X, int64_t M, int64_t K, const int8_t* Wq8,
                      const uint16_t* sw16, int64_t N, double* Y)
{
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double s = (double)oracle_half_to_float(sw16[n]);
            double y = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double w = (double)Wq8[n * K + k] * s;
                y += w * (double)oracle_half_to_float(X[m * K + k]);
            }
            Y[m * N + n] = y;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* g1: group-wise INT4 weight quantizer  [P1 后续优化方向: group-wise scale,  */
/*     the row-wise definition of 当前实现方式 applied to each group of a row] */
/* ------------------------------------------------------------------------ */

/* Floats per row of the group-scale matrix: K / gs rounded up to a multiple
   of 4, so that every scale row starts on a 16-byte boundary.  The pages fix
   no storage layout; this is the library's documented one. */
int64_t oracle_w4g_scale_stride(int64_t K, int64_t gs)
{
    if (gs <= 0 || K < 0) return 0;
    int64_t groups = K / gs;
    return (groups + 3) / 4 * 4;
}

/* W[N][K] fp32 -> Wq[N][K/2] packed nibbles (same packing as the row-wise
   quantizer) + sg[N][stride] fp32.  Group g of row n covers the codes
   k = g*gs .. g*gs+gs-1; its scale is s = max|W over the group| / 7 and its
   codes q = clamp(round(W / s), -7, 7).  Padding entries of sg are 0.
   With gs == K this is the row-wise quantizer. */
int oracle_w4g_quantize(const float* W, int64_t N, int64_t K, int64_t gs, uint8_t* Wq,
                        float* sg)
{
    if (N < 0 || K < 0 || gs < 2 || (gs & 1) || K % gs) return ORACLE_ERR_SHAPE;
    int64_t groups = K / gs;
    int64_t ld = oracle_w4g_scale_stride(K, gs);
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t g = 0; g < ld; ++g) {
            if (g >= groups) {
                sg[n * ld + g] = 0.0f;
                continue;
            }
            const float* grp = W + n * K + g * gs;
            float s = row_absmax(grp, gs) / 7.0f;
            sg[n * ld + g] = s;
            for (int64_t j = 0; j < gs / 2; ++j) {
                int q0 = quant_code(grp[2 * j], s, 7);
                int q1 = quant_code(grp[2 * j + 1], s, 7);
                Wq[n * (K / 2) + g * (gs / 2) + j] = (uint8_t)((q0 & 0xF) | ((q1 & 0xF) << 4));
            }
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* g2: group-wise W4A8 product, binary64 reference  [P1 当前实现方式: output */
/*     = int32 accumulate * weight_scale * activation_scale, per group]      */
/* ------------------------------------------------------------------------ */

/* For every (m, n):
     acc_g = sum over group g of Xq[m][k] * q_w[n][k]          (int64, exact)
     Y[m][n] = s_a[m] * sum_g s_g[n][g] * acc_g                (binary64)
     B[m][n] = s_a[m] * sum_g s_g[n][g] * sum over g of |Xq * q_w|
   B is the magnitude in which the rounding error of an fp32 evaluation of Y
   is bounded.  Every product s_g * acc_g is exact in binary64 (a 24-bit
   significand times an integer below 2^26 for gs <= 2^16); only the sums
   and the final product round. */
int oracle_w4a8g_ref(const int8_t* Xq, const float* sa, int64_t M, int64_t K, int64_t gs,
                     const uint8_t* Wq, const float* sg, int64_t N, double* Y, double* B)
{
    if (M < 0 || N < 0 || K < 0 || gs < 2 || (gs & 1) || K % gs || gs > 65536)
        return ORACLE_ERR_SHAPE;
    int64_t groups = K / gs;
    int64_t ld = oracle_w4g_scale_stride(K, gs);
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double y = 0.0, b = 0.0;
            for (int64_t g = 0; g < groups; ++g) {
                int64_t acc = 0, mag = 0;
                for (int64_t j = g * (gs / 2); j < (g + 1) * (gs / 2); ++j) {
                    uint8_t byte = Wq[n * (K / 2) + j];
                    int64_t p0 = (int64_t)Xq[m * K + 2 * j] * nibble_value(byte & 0xFu);
                    int64_t p1 = (int64_t)Xq[m * K + 2 * j + 1] * nibble_value(byte >> 4);
                    acc += p0 + p1;
                    mag += (p0 < 0 ? -p0 : p0) + (p1 < 0 ? -p1 : p1);
                }
                double s = (double)sg[n * ld + g];
                y += s * (double)acc;
                b += s * (double)mag;
            }
            Y[m * N + n] = (double)sa[m] * y;
            B[m * N + n] = (double)sa[m] * b;
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* g3: group-wise W4A8 product in binary32, in the library's fixed order     */
/*     [P1 当前实现方式: int32 accumulate times the weight scale times the    */
/*     activation scale, applied per group as 后续优化方向 suggests]          */
/* ------------------------------------------------------------------------ */

/* The page gives the arithmetic but no summation order for the per-group
   products, and an fp32 sum depends on its order.  This is the order the
   library fixes (a function of K and gs only, never of a launch plan):
     acc_g   = exact integer sum of group g (as in g2), converted to binary32
               with one round-to-nearest (exact for gs <= 16384)
     L       = max(gs, 1024) codes: the fold chunk; chunk c holds the
               groups whose codes lie in [c*L, (c+1)*L)
     f_c     = +0, then for every group g of chunk c in ascending order
               f_c = fmaf(acc_g, s_g, f_c)         (one rounding each)
     F       = +0, then for every chunk c in ascending order F = F + f_c
     Y[m][n] = F * s_a[m]
   fmaf is C99's fused multiply-add (a single IEEE rounding); the other
   operations are single binary32 operations (no contraction).  Chunks let
   the K dimension be split at chunk boundaries without changing a bit. */
int oracle_w4a8g_f32(const int8_t* Xq, const float* sa, int64_t M, int64_t K, int64_t gs,
                     const uint8_t* Wq, const float* sg, int64_t N, float* Y)
{
    if (M < 0 || N < 0 || K < 0 || gs < 2 || (gs & 1) || K % gs || gs > 65536)
        return ORACLE_ERR_SHAPE;
    int64_t ld = oracle_w4g_scale_stride(K, gs);
    int64_t L = gs > 1024 ? gs : 1024;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            float F = 0.0f;
            for (int64_t c0 = 0; c0 < K; c0 += L) {
                int64_t c1 = c0 + L < K ? c0 + L : K;
                float f = 0.0f;
                for (int64_t k0 = c0; k0 < c1; k0 += gs) {
                    int64_t acc = 0;
                    for (int64_t j = k0 / 2; j < (k0 + gs) / 2; ++j) {
                        uint8_t byte = Wq[n * (K / 2) + j];
                        acc += (int64_t)Xq[m * K + 2 * j] * nibble_value(byte & 0xFu);
                        acc += (int64_t)Xq[m * K + 2 * j + 1] * nibble_value(byte >> 4);
                    }
                    f = fmaf((float)acc, sg[n * ld + k0 / gs], f);
                }
                F = F + f;
            }
            Y[m * N + n] = F * sa[m];
        }
    }
    return ORACLE_OK;
}

/* The whole group-wise linear in the fixed binary32 order: the activation
   quantizer of a2, then g3. */
int oracle_w4a8g_linear_f32(const uint16_t* X, int64_t M, int64_t K, int64_t gs,
                            const uint8_t* Wq, const float* sg, int64_t N, float* Y,
                            int8_t* Xq_out, float* sa_out)
{
    int st = oracle_act_quantize(X, M, K, Xq_out, sa_out);
    if (st != ORACLE_OK) return st;
    return oracle_w4a8g_f32(Xq_out, sa_out, M, K, gs, Wq, sg, N, Y);
}

/* The whole group-wise linear: the per-row activation quantizer of a2, then
   the reference above. */
int oracle_w4a8g_linear(const uint16_t* X, int64_t M, int64_t K, int64_t gs, const uint8_t* Wq,
                        const float* sg, int64_t N, double* Y, double* B, int8_t* Xq_out,
                        float* sa_out)
{
    int st = oracle_act_quantize(X, M, K, Xq_out, sa_out);
    if (st != ORACLE_OK) return st;
    return oracle_w4a8g_ref(Xq_out, sa_out, M, K, gs, Wq, sg, N, Y, B);
}

/* ------------------------------------------------------------------------ */
/* s1-s3: IndexSoftmax  [P3 "IntAttention: 全整数注意力流水线", section     */
/*        基准/方法设计: IndexSoftmax 的三个机制]                            */
/* ------------------------------------------------------------------------ */
/* Readings where the page leaves a step open: the rounding bracket of every
   formula is round to nearest with halves away from zero (all operands are
   non-negative, so halves go up); LUT entries and c_int are computed in
   binary64 with the C library's exp and sqrt; a row whose c_int is 0 clips
   every distance to 0 and takes index 0 everywhere. */

/* Mechanism 2: the 2^b-entry exponent table quantized to UINT8,
   LUT[i] = round(255 * exp(-c * i / (2^b - 1))), the last entry forced to 0. */
int oracle_isx_lut(int b, double c, uint8_t* lut)
{
    if (b < 1 || b > 8 || !(c > 0.0)) return ORACLE_ERR_SHAPE;
    int n = 1 << b;
    for (int i = 0; i < n - 1; ++i)
        lut[i] = (uint8_t)round(255.0 * exp(-c * (double)i / (double)(n - 1)));
    lut[n - 1] = 0;
    return ORACLE_OK;
}

/* Mechanism 1's clipping threshold in integer logit units:
   c_int = round(c * sqrt(d) / (s_Q * s_K)). */
int64_t oracle_isx_c_int(double c, int64_t d, float s_q, float s_k)
{
    return (int64_t)llround(c * sqrt((double)d) / ((double)s_q * (double)s_k));
}

/* IndexSoftmax of the int32 logits A[rows][cols] into UINT8 probabilities
   P[rows][cols], per row:
     delta  = rowMax(A) - A                        (mechanism 1)
     delta' = min(delta, c_int)
     idx    = round(delta' * (2^b - 1) / c_int)    (mechanism 2)
     E      = LUT[idx]
     P      = round(255 * E / rowSum(E))           (mechanism 3)
   All arithmetic is exact integer arithmetic (int64). */
int oracle_index_softmax(const int32_t* A, int64_t rows, int64_t cols, int64_t c_int, int b,
                         const uint8_t* lut, uint8_t* P)
{
    if (rows < 0 || cols < 1 || c_int < 0 || b < 1 || b > 8) return ORACLE_ERR_SHAPE;
    int64_t top = (1 << b) - 1;
    for (int64_t r = 0; r < rows; ++r) {
        const int32_t* a = A + r * cols;
        int32_t mx = a[0];
        for (int64_t k = 1; k < cols; ++k)
            if (a[k] > mx) mx = a[k];
        int64_t sum = 0;
        for (int64_t k = 0; k < cols; ++k) {
            int64_t delta = (int64_t)mx - (int64_t)a[k];
            int64_t clipped = delta < c_int ? delta : c_int;
            /* round(clipped * top / c_int), halves up: floor((2 x top + c) / 2c) */
            int64_t idx = c_int > 0 ? (2 * clipped * top + c_int) / (2 * c_int) : 0;
            sum += lut[idx];
        }
        for (int64_t k = 0; k < cols; ++k) {
            int64_t delta = (int64_t)mx - (int64_t)a[k];
            int64_t clipped = delta < c_int ? delta : c_int;
            int64_t idx = c_int > 0 ? (2 * clipped * top + c_int) / (2 * c_int) : 0;
            int64_t e = lut[idx];
            /* round(255 e / sum), halves up; sum >= LUT[0] = 255 > 0 */
            P[r * cols + k] = (uint8_t)((2 * 255 * e + sum) / (2 * sum));
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* The MLP's gated product between gate/up and down                          */
/* ------------------------------------------------------------------------ */

/* binary64 -> binary16, round to nearest, ties to even, written from the
   format's definition: the result's quantum is 2^(eh - 10) with
   eh = max(floor(log2 |x|), -14) (subnormals share eh = -14); |x| / quantum
   is an exact scaling, rounded once by rint (ties to even); a carry to 2048
   moves to the next exponent, past 65504 (half an ulp included) to inf. */
uint16_t oracle_double_to_half(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7E00u);
    double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7C00u);
    if (a == 0.0) return sign;
    int e;
    (void)frexp(a, &e);                  /* a = f * 2^e, f in [0.5, 1) */
    int eh = e - 1 < -14 ? -14 : e - 1;  /* floor(log2 a), clamped */
    if (eh > 15) return (uint16_t)(sign | 0x7C00u);
    double n = rint(ldexp(a, 10 - eh));  /* a / 2^(eh - 10): exact, then one rounding */
    /* n = 2048 carries into the exponent; at eh = 15 that is 0x7C00 = inf */
    uint32_t bits = (eh == -14) ? (uint32_t)n : ((uint32_t)(eh + 15) << 10) + ((uint32_t)n - 1024u);
    return (uint16_t)(sign | bits);
}

/* The gated product that the MLP of the INT4 page's model (a Qwen2-7B,
   HIDDEN 3584 / INTERMEDIATE 18944: gate and up projections, then down)
   feeds to the down projection, whose activation quantization the page's
   section 后续优化方向 asks to make cheaper.  The pages do not print the
   activation; the reading is that model family's SwiGLU:
     v = silu(g) * u = g / (1 + exp(-g)) * u      in binary64 (exact inputs),
     h = binary16(v)                               rounded to nearest even,
   for i < n.  v is returned too, for the rounding-boundary check. */
void oracle_silu_mul(const float* g, const float* u, int64_t n, double* v, uint16_t* h)
{
    for (int64_t i = 0; i < n; ++i) {
        double x = (double)g[i];
        double p = x / (1.0 + exp(-x)) * (double)u[i];
        v[i] = p;
        h[i] = oracle_double_to_half(p);
    }
}
