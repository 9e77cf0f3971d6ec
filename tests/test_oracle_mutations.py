"""Plant plausible mistakes in copies of the oracle (on the CPU) and check that
at least one pin catches each.  This is what makes the pins a check of the
oracle rather than a restatement of it."""
import os

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(os.path.abspath(oracle.__file__)), "oracle.c")

# (name, exact text in oracle.c, replacement)
MUTATIONS = [
    ("round_half_even", "float r = roundf(t);", "float r = rintf(t);"),
    ("round_toward_zero", "float r = roundf(t);", "float r = truncf(t);"),
    ("reciprocal_multiply", "float t = v / s;", "float t = v * (1.0f / s);"),
    ("nibble_order_pack",
     "(uint8_t)((q0 & 0xF) | ((q1 & 0xF) << 4))", "(uint8_t)((q1 & 0xF) | ((q0 & 0xF) << 4))"),
    ("nibble_unsigned", "return v >= 8 ? (int)v - 16 : (int)v;", "return (int)v;"),
    ("nibble_sign_offset", "return v >= 8 ? (int)v - 16 : (int)v;", "return v >= 8 ? (int)v - 15 : (int)v;"),
    ("w4_divisor_8", "row_absmax(row, K) / 7.0f", "row_absmax(row, K) / 8.0f"),
    ("act_divisor_128", "float s = mx / 127.0f;", "float s = mx / 128.0f;"),
    ("absmax_without_abs", "float a = fabsf(row[k]);", "float a = row[k];"),
    ("act_row_index", "quant_code(oracle_half_to_float(X[m * K + k]), s, 127)",
     "quant_code(oracle_half_to_float(X[k]), s, 127)"),
    ("dot_nibble_swap",
     "s += (int64_t)Xq[m * K + 2 * j] * nibble_value(b & 0xFu);\n"
     "                s += (int64_t)Xq[m * K + 2 * j + 1] * nibble_value(b >> 4);",
     "s += (int64_t)Xq[m * K + 2 * j] * nibble_value(b >> 4);\n"
     "                s += (int64_t)Xq[m * K + 2 * j + 1] * nibble_value(b & 0xFu);"),
    ("dot_dropped_high", "s += (int64_t)Xq[m * K + 2 * j + 1] * nibble_value(b >> 4);", ""),
    ("dot_transposed_act", "(int64_t)Xq[m * K + 2 * j]", "(int64_t)Xq[n * K + 2 * j]"),
    ("rescale_swapped_index", "float t = (float)acc[m * N + n] * sw[n];\n            Y[m * N + n] = t * sa[m];",
     "float t = (float)acc[m * N + n] * sa[m];\n            Y[m * N + n] = t * sw[n];"),
    ("rescale_dropped_sa", "Y[m * N + n] = t * sa[m];", "Y[m * N + n] = t;"),
    ("rescale_sw_row_index", "* sw[n];", "* sw[m];"),
    ("clamp_dropped", "if (r > (float)qmax) r = (float)qmax;", ""),
    ("w8_unrounded_scale", "float s = oracle_half_to_float(h);", "float s = row_absmax(row, K) / 127.0f;"),
    ("w8a16_scale_twice", "double w = (double)Wq8[n * K + k] * s;", "double w = (double)Wq8[n * K + k] * s * s;"),
    ("w8a16_scale_dropped", "double w = (double)Wq8[n * K + k] * s;", "double w = (double)Wq8[n * K + k];"),
    ("half_subnormal_exponent", "v = ldexpf((float)m, -24);", "v = ldexpf((float)m, -25);"),
    ("half_normal_bias", "ldexpf((float)(1024 + m), e - 25)", "ldexpf((float)(1024 + m), e - 24)"),
    ("half_encode_ties_up", "if (rem > half || (rem == half && (n & 1u))) n += 1;", "if (rem >= half) n += 1;"),
    ("half_encode_truncate", "if (rem > half || (rem == half && (n & 1u))) n += 1;", ""),
    ("half_encode_overflow", "if (bits >= 0x7C00u) bits = 0x7C00u;", ""),
    ("w4g_row_max", "float s = row_absmax(grp, gs) / 7.0f;", "float s = row_absmax(W + n * K, K) / 7.0f;"),
    ("w4g_divisor_8", "row_absmax(grp, gs) / 7.0f", "row_absmax(grp, gs) / 8.0f"),
    ("w4g_pack_group_offset", "Wq[n * (K / 2) + g * (gs / 2) + j]", "Wq[n * (K / 2) + j]"),
    ("w4g_stride_unpadded", "return (groups + 3) / 4 * 4;", "return groups;"),
    ("w4g_ref_scale_group0", "double s = (double)sg[n * ld + g];", "double s = (double)sg[n * ld];"),
    ("w4g_ref_dropped_sa", "Y[m * N + n] = (double)sa[m] * y;", "Y[m * N + n] = y;"),
    ("w4g_ref_signed_magnitude", "mag += (p0 < 0 ? -p0 : p0) + (p1 < 0 ? -p1 : p1);", "mag += p0 + p1;"),
    ("w4g_ref_group_bytes", "for (int64_t j = g * (gs / 2); j < (g + 1) * (gs / 2); ++j)",
     "for (int64_t j = 0; j < gs / 2; ++j)"),
    ("w4g_ref_dropped_high", "acc += p0 + p1;", "acc += p0;"),
    ("w4g_f32_descending", "for (int64_t k0 = c0; k0 < c1; k0 += gs) {",
     "for (int64_t k0 = c1 - gs; k0 >= c0; k0 -= gs) {"),
    ("w4g_f32_unfused", "f = fmaf((float)acc, sg[n * ld + k0 / gs], f);",
     "f = f + (float)acc * sg[n * ld + k0 / gs];"),
    ("w4g_f32_unchunked", "int64_t L = gs > 1024 ? gs : 1024;", "int64_t L = K > 0 ? K : 1;"),
    ("w4g_f32_chunk_512", "int64_t L = gs > 1024 ? gs : 1024;", "int64_t L = gs > 512 ? gs : 512;"),
    ("w4g_f32_dropped_chunks", "F = F + f;", "F = f;"),
    ("w4g_f32_dropped_sa", "Y[m * N + n] = F * sa[m];", "Y[m * N + n] = F;"),
    ("w4g_f32_scale_group0", "sg[n * ld + k0 / gs], f);", "sg[n * ld], f);"),
    ("w4g_f32_dropped_high", "acc += (int64_t)Xq[m * K + 2 * j + 1] * nibble_value(byte >> 4);", ""),
    ("silu_sign_of_exp", "double p = x / (1.0 + exp(-x)) * (double)u[i];", "double p = x / (1.0 + exp(x)) * (double)u[i];"),
    ("silu_dropped_up", "double p = x / (1.0 + exp(-x)) * (double)u[i];", "double p = x / (1.0 + exp(-x));"),
    ("silu_sigmoid_only", "double p = x / (1.0 + exp(-x)) * (double)u[i];", "double p = 1.0 / (1.0 + exp(-x)) * (double)u[i];"),
    ("silu_half_via_float", "h[i] = oracle_double_to_half(p);", "h[i] = oracle_float_to_half((float)p);"),
    ("d2h_truncate", "double n = rint(ldexp(a, 10 - eh));", "double n = floor(ldexp(a, 10 - eh));"),
    ("d2h_ties_away", "double n = rint(ldexp(a, 10 - eh));", "double n = round(ldexp(a, 10 - eh));"),
    ("d2h_subnormal_exponent", "int eh = e - 1 < -14 ? -14 : e - 1;", "int eh = e - 1 < -15 ? -15 : e - 1;"),
    ("d2h_overflow_threshold", "if (eh > 15) return (uint16_t)(sign | 0x7C00u);", "if (eh > 16) return (uint16_t)(sign | 0x7C00u);"),
    ("isx_lut_scale_254", "(uint8_t)round(255.0 * exp(", "(uint8_t)round(254.0 * exp("),
    ("isx_lut_step_2b", "exp(-c * (double)i / (double)(n - 1))", "exp(-c * (double)i / (double)n)"),
    ("isx_lut_last_not_zero", "lut[n - 1] = 0;", "lut[n - 1] = (uint8_t)round(255.0 * exp(-c));"),
    ("isx_c_int_without_sqrt", "c * sqrt((double)d) /", "c * (double)d /"),
    ("isx_c_int_truncated", "(int64_t)llround(c * sqrt", "(int64_t)(c * sqrt"),
    ("isx_idx_floor", "(2 * clipped * top + c_int) / (2 * c_int)", "(clipped * top) / c_int"),
    ("isx_sum_counts", "sum += lut[idx];", "sum += 255;"),
    ("isx_p_floor", "(2 * 255 * e + sum) / (2 * sum)", "(255 * e) / sum"),
    ("isx_p_scale_256", "(2 * 255 * e + sum) / (2 * sum)", "(2 * 256 * e + sum) / (2 * sum)"),
]


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutation_is_caught(tmp_path, source, name, old, new):
    assert source.count(old) >= 1, "mutation %s no longer matches oracle.c" % name
    path = tmp_path / "oracle_mut.c"
    path.write_text(source.replace(old, new))
    lib = oracle.compile_oracle(str(path), str(tmp_path / "liboracle_mut.so"))
    mut = oracle.Oracle(lib)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(mut)
        except (AssertionError, ValueError, OverflowError, IndexError):
            caught.append(pin.__name__)
            break
    assert caught, "planted mistake %r passed every pin" % name
