"""Pins for the CPU oracle: checks against what the pages and mathematics fix.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with something other than itself: hand-derived
closed forms from ``tests/golden/``, sizes printed on the pages, exhaustive
comparisons with numpy's IEEE binary16 conversion, exact rational arithmetic,
numpy integer/fp64 matrix products on decoded codes, invariants of
round-to-nearest quantization and a deterministic end-to-end error bound.

The same functions run against deliberately broken copies of ``oracle.c`` in
``test_oracle_mutations.py``: every planted mistake must trip at least one pin.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------

def read_cases(name):
    """Parse a golden file made of ``case <name>`` blocks of ``key: values``."""
    cases, cur = [], None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if line.startswith("case "):
                cur = {"name": line[5:].strip()}
                cases.append(cur)
            else:
                key, val = line.split(":", 1)
                cur[key.strip()] = val.split()
    return cases


def read_kv(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split(":", 1)
                out[k.strip()] = float(v)
    return out


def f32_nearest(fr: Fraction) -> np.float32:
    """Exact round-to-nearest-even of a rational into binary32 (normal range)."""
    if fr == 0:
        return np.float32(0.0)
    neg = fr < 0
    a = -fr if neg else fr
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    assert -126 <= e <= 127
    scaled = a / Fraction(2) ** (e - 23)          # in [2^23, 2^24)
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    v = math.ldexp(float(n), e - 23)
    return np.float32(-v if neg else v)


def round_half_away(v: float) -> int:
    a = abs(v)
    r = math.floor(a + 0.5) if a - math.floor(a) != 0.5 else math.floor(a) + 1
    return int(math.copysign(r, v)) if r else 0


def decode_nibbles(Wq: np.ndarray) -> np.ndarray:
    """Independent decode used only to feed numpy products (pinned by golden bytes)."""
    lo = (Wq & 0x0F).astype(np.int16)
    hi = (Wq >> 4).astype(np.int16)
    lo = np.where(lo >= 8, lo - 16, lo)
    hi = np.where(hi >= 8, hi - 16, hi)
    out = np.empty((Wq.shape[0], Wq.shape[1] * 2), np.int64)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    return out


# --------------------------------------------------------------------------
# binary16
# --------------------------------------------------------------------------

def pin_half_decode_exhaustive(o):
    """All 65536 binary16 patterns decode exactly as numpy's IEEE conversion."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([o.half_to_float(int(b)) for b in bits], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def pin_half_encode(o):
    """Round-to-nearest-even float->binary16 agrees with numpy on edge values
    (ties, overflow threshold, subnormal boundaries) and random bit patterns."""
    edges = [0.0, -0.0, 1.0, 65504.0, 65519.996, 65520.0, 65536.0, 1e9, -65520.0,
             2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -26, 2.0 ** -14,
             2.0 ** -14 - 2.0 ** -25, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11,
             2049.0, 2051.0, 1e-30, -1e-30, float("inf"), -float("inf"), 5.9604645e-08,
             8.940697e-08, 0.33325195, 1.0 / 3.0]
    rng = np.random.Generator(np.random.PCG64(12345))
    rand_bits = rng.integers(0, 2 ** 32, size=60000, dtype=np.uint64).astype(np.uint32)
    # bias the random set towards the binary16 range (exponents 100..150)
    near = (rng.integers(100, 150, size=60000).astype(np.uint32) << 23) | (
        rng.integers(0, 2 ** 23, size=60000).astype(np.uint32)) | (
        rng.integers(0, 2, size=60000).astype(np.uint32) << 31)
    vals = np.concatenate([np.array(edges, np.float32), rand_bits.view(np.float32),
                           near.view(np.float32)])
    with np.errstate(over="ignore", invalid="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([o.float_to_half(float(v)) for v in vals], dtype=np.uint16)
    nan = np.isnan(vals)
    assert np.all((got[nan] & 0x7C00) == 0x7C00) and np.all((got[nan] & 0x3FF) != 0)
    bad = np.nonzero(got[~nan] != ref[~nan])[0]
    assert bad.size == 0, "first mismatch at %r" % (vals[~nan][bad[:3]],)


# --------------------------------------------------------------------------
# a1: INT4 weight quantizer and packing
# --------------------------------------------------------------------------

def pin_w4_golden(o):
    """Hand-derived closed forms: scale, codes, packed bytes, decode."""
    for c in read_cases("w4_quant_closed_forms.txt"):
        row = np.array([float(v) for v in c["row"]], np.float32)[None, :]
        Wq, sw = o.w4_quantize(row)
        assert sw[0] == np.float32(float(c["scale"][0])), c["name"]
        want = np.array([int(b, 16) for b in c["bytes"]], np.uint8)
        assert np.array_equal(Wq[0], want), (c["name"], Wq[0], want)
        codes = np.array([int(v) for v in c["codes"]], np.int8)
        assert np.array_equal(o.w4_unpack(Wq, row.shape[1])[0], codes), c["name"]


def pin_w4_all_code_pairs(o):
    """Every pair of codes in [-7, 7] survives quantize -> pack -> unpack, and
    the byte equals the two's-complement nibbles, low nibble first."""
    codes = np.array([(a, b) for a in range(-7, 8) for b in range(-7, 8)], np.int64).ravel()
    row = np.concatenate([[7.0], codes.astype(np.float64), [0.0]]).astype(np.float32)[None, :]
    Wq, sw = o.w4_quantize(row)
    assert sw[0] == 1.0
    q = o.w4_unpack(Wq, row.shape[1])[0]
    assert np.array_equal(q[1:-1], codes)
    # byte j holds codes 2j (low) and 2j+1 (high); shift by one for the leading 7
    b = Wq[0]
    assert np.array_equal(decode_nibbles(Wq)[0], q.astype(np.int64))
    lows = [(int(v) & 0xF) for v in q[0::2]]
    highs = [(int(v) & 0xF) for v in q[1::2]]
    assert list(b) == [lo | (hi << 4) for lo, hi in zip(lows, highs)]


def pin_w4_true_division(o):
    """Codes follow round(fl(w / s)) with a correctly rounded IEEE quotient,
    checked in exact rational arithmetic on near-tie inputs."""
    rng = np.random.Generator(np.random.PCG64(7))
    rows = []
    for _ in range(400):
        mx = np.float32(rng.uniform(0.01, 1.0))
        s = f32_nearest(Fraction(float(mx)) / 7)
        r = [mx]
        for k in range(-6, 7):
            t = Fraction(2 * k + 1, 2)  # a .5 tie of the quotient
            w = np.float32(float(t * Fraction(float(s))))
            for d in (-2, -1, 0, 1, 2):
                v = w
                for _ in range(abs(d)):
                    v = np.nextafter(v, np.float32(np.inf if d > 0 else -np.inf), dtype=np.float32)
                r.append(v)
        rows.append(r[:64] if len(r) >= 64 else r + [0.0] * (64 - len(r)))
    W = np.array(rows, np.float32)
    Wq, sw = o.w4_quantize(W)
    q = o.w4_unpack(Wq, W.shape[1])
    for n in range(W.shape[0]):
        s = Fraction(float(sw[n]))
        assert sw[n] == f32_nearest(Fraction(float(np.max(np.abs(W[n])))) / 7)
        for k in range(W.shape[1]):
            t = f32_nearest(Fraction(float(W[n, k])) / s) if W[n, k] != 0 else np.float32(0)
            want = max(-7, min(7, round_half_away(float(t))))
            assert q[n, k] == want, (n, k, float(W[n, k]), float(sw[n]), q[n, k], want)


def pin_w4_invariants(o):
    """On seeded N(0, 0.02) rows (with a few x20 outliers): |w - q*s| <= s/2,
    the row's largest |w| gets code +-7 with its sign, codes stay in [-7, 7]."""
    W = synth.normal(11, (48, 896), 0.02)
    W[5, 100] *= 20.0
    W[9, :] = 0.0
    W[17, 3] = -0.5
    Wq, sw = o.w4_quantize(W)
    q = o.w4_unpack(Wq, W.shape[1]).astype(np.float64)
    s = sw.astype(np.float64)[:, None]
    err = np.abs(W.astype(np.float64) - q * s)
    assert np.all(err <= s / 2 * (1 + 2 ** -20) + 1e-45)
    assert np.all(np.abs(q) <= 7)
    for n in range(W.shape[0]):
        if sw[n] == 0:
            assert not W[n].any() and not q[n].any()
            continue
        k = int(np.argmax(np.abs(W[n])))
        assert q[n, k] == 7 * np.sign(W[n, k])
        assert abs(float(sw[n]) * 7 - float(np.max(np.abs(W[n])))) <= 4e-7 * float(np.max(np.abs(W[n])))


# --------------------------------------------------------------------------
# a2: activation quantizer
# --------------------------------------------------------------------------

def pin_act_golden(o):
    for c in read_cases("act_quant_closed_forms.txt"):
        x = np.array([float(v) for v in c["x"]], np.float16)[None, :]
        assert np.array_equal(x.astype(np.float64)[0], [float(v) for v in c["x"]])
        Xq, sa = o.act_quantize(x)
        assert sa[0] == np.float32(float(c["scale"][0])), c["name"]
        assert np.array_equal(Xq[0], np.array([int(v) for v in c["codes"]], np.int8)), c["name"]


def pin_act_invariants(o):
    """|x - q*s_a| <= s_a/2, max |x| -> +-127, codes within [-127, 127], per row."""
    X = synth.activation(21, 6, 3584, outlier_frac=0.001)
    X[2] = 0
    Xq, sa = o.act_quantize(X)
    x = X.astype(np.float64)
    s = sa.astype(np.float64)[:, None]
    assert np.all(np.abs(x - Xq.astype(np.float64) * s) <= s / 2 * (1 + 2 ** -20) + 1e-45)
    assert np.all(np.abs(Xq.astype(np.int64)) <= 127)
    for m in range(X.shape[0]):
        if sa[m] == 0:
            assert not Xq[m].any()
            continue
        k = int(np.argmax(np.abs(x[m])))
        assert Xq[m, k] == 127 * np.sign(x[m, k])
        assert sa[m] == f32_nearest(Fraction(float(np.max(np.abs(x[m])))) / 127)


# --------------------------------------------------------------------------
# a3+a4: integer dot
# --------------------------------------------------------------------------

def pin_dot_closed_forms(o):
    K = 96
    W = np.full((2, K // 2), 0x77, np.uint8)          # every code +7
    X = np.full((1, K), 127, np.int8)
    assert np.all(o.w4a8_dot(X, W) == 889 * K)
    X2 = np.tile(np.array([127, -127], np.int8), K // 2)[None, :]
    assert np.all(o.w4a8_dot(X2, W) == 0)
    # asymmetric byte: low code 7, high code 1; activation only on even k
    W3 = np.full((1, K // 2), 0x17, np.uint8)
    X3 = np.tile(np.array([1, 0], np.int8), K // 2)[None, :]
    assert o.w4a8_dot(X3, W3)[0, 0] == 7 * (K // 2)
    X4 = np.tile(np.array([0, 1], np.int8), K // 2)[None, :]
    assert o.w4a8_dot(X4, W3)[0, 0] == 1 * (K // 2)
    # one-hot activations recover every code at its index
    W5 = np.frombuffer(bytes(range(0, 256, 3))[:K // 2], np.uint8)[None, :].copy()
    q = decode_nibbles(W5)[0]
    for k in range(K):
        e = np.zeros((1, K), np.int8)
        e[0, k] = -127
        assert o.w4a8_dot(e, W5)[0, 0] == -127 * q[k]
    # extreme magnitudes: -8 codes (legal on input) with -127 activations
    W6 = np.full((1, K // 2), 0x88, np.uint8)
    assert o.w4a8_dot(np.full((1, K), -127, np.int8), W6)[0, 0] == 8 * 127 * K


def pin_dot_bruteforce(o):
    """acc equals numpy's int64 matrix product of the decoded codes."""
    for (M, N, K, seed) in [(1, 7, 64, 1), (3, 5, 32, 2), (4, 9, 160, 3)]:
        W = synth.normal(seed, (N, K), 0.02)
        Wq, _ = o.w4_quantize(W)
        Xq, _ = o.act_quantize(synth.activation(seed + 100, M, K))
        ref = Xq.astype(np.int64) @ decode_nibbles(Wq).T
        assert np.array_equal(o.w4a8_dot(Xq, Wq).astype(np.int64), ref)


# --------------------------------------------------------------------------
# a5: rescale
# --------------------------------------------------------------------------

def pin_rescale_powers_of_two(o):
    """With power-of-two scales the result is exact: Y[m][n] = acc * 2^-(n+3) * 2^-(4m)."""
    M, N = 3, 6
    acc = (np.arange(M * N, dtype=np.int64).reshape(M, N) * 7919 - 40000).astype(np.int32)
    sw = np.array([2.0 ** -(n + 3) for n in range(N)], np.float32)
    sa = np.array([2.0 ** -(4 * m) for m in range(M)], np.float32)
    Y = o.w4a8_rescale(acc, sw, sa)
    want = np.array([[acc[m, n] * 2.0 ** -(n + 3) * 2.0 ** -(4 * m) for n in range(N)]
                     for m in range(M)])
    assert np.array_equal(Y.astype(np.float64), want)


def pin_rescale_order(o):
    """The fixed contract: (float(acc) * s_w) * s_a, each product rounded to
    binary32; checked with exact rationals on values where orders differ."""
    rng = np.random.Generator(np.random.PCG64(3))
    acc = rng.integers(-2 ** 30, 2 ** 30, size=(4, 64)).astype(np.int32)
    sw = rng.uniform(1e-4, 1e-2, size=64).astype(np.float32)
    sa = rng.uniform(1e-3, 1.0, size=4).astype(np.float32)
    Y = o.w4a8_rescale(acc, sw, sa)
    differs = 0
    for m in range(4):
        for n in range(64):
            a = f32_nearest(Fraction(int(acc[m, n])))
            t = f32_nearest(Fraction(float(a)) * Fraction(float(sw[n])))
            y = f32_nearest(Fraction(float(t)) * Fraction(float(sa[m])))
            assert Y[m, n] == y
            other = f32_nearest(Fraction(float(a)) *
                                Fraction(float(f32_nearest(Fraction(float(sw[n])) * Fraction(float(sa[m]))))))
            differs += int(other != y)
    assert differs > 0  # the inputs do separate the two orders


# --------------------------------------------------------------------------
# a-f: end to end
# --------------------------------------------------------------------------

def pin_linear_error_bound(o):
    """Quantized linear vs fp64 unquantized GEMV within the deterministic bound
    sum_k(|w| s_a/2 + |x| s_w/2 + 3 s_w s_a/4)(1+2^-18) + 3*2^-24 |Y|."""
    for (M, N, K, seed) in [(1, 64, 896, 5), (2, 16, 3584, 6)]:
        W = synth.normal(seed, (N, K), 0.02)
        X = synth.activation(seed + 50, M, K, outlier_frac=0.001)
        Wq, sw = o.w4_quantize(W)
        Y, Xq, sa, acc = o.w4a8_linear(X, Wq, sw)
        ref = X.astype(np.float64) @ W.astype(np.float64).T
        s_w = sw.astype(np.float64)[None, :]
        s_a = sa.astype(np.float64)[:, None]
        bound = ((np.abs(X).astype(np.float64).sum(1)[:, None] * s_w / 2
                  + np.abs(W).astype(np.float64).sum(1)[None, :] * s_a / 2
                  + K * 3 * s_w * s_a / 4) * (1 + 2 ** -18) + 3 * 2.0 ** -24 * np.abs(Y))
        assert np.all(np.abs(Y.astype(np.float64) - ref) <= bound)
        # sanity: row-wise INT4 keeps the output's direction (measured ~0.985)
        cos = float((Y.astype(np.float64) * ref).sum() /
                    np.sqrt((Y.astype(np.float64) ** 2).sum() * (ref ** 2).sum()))
        assert cos > 0.97


# --------------------------------------------------------------------------
# g1/g2: group-wise INT4 scales
# --------------------------------------------------------------------------

def pin_w4g_golden(o):
    """Hand-derived closed forms: per-group scales (with the zero padding of
    the scale row), codes and packed bytes."""
    for c in read_cases("w4g_quant_closed_forms.txt"):
        gs = int(c["gs"][0])
        row = np.array([float(v) for v in c["row"]], np.float32)[None, :]
        Wq, sg = o.w4g_quantize(row, gs)
        want_s = np.array([float(v) for v in c["scales"]], np.float32)
        assert np.array_equal(sg[0], want_s), (c["name"], sg[0], want_s)
        want = np.array([int(b, 16) for b in c["bytes"]], np.uint8)
        assert np.array_equal(Wq[0], want), (c["name"], Wq[0], want)
        codes = np.array([int(v) for v in c["codes"]], np.int64)
        assert np.array_equal(decode_nibbles(Wq)[0], codes), c["name"]


def pin_w4g_scale_stride(o):
    """Scale rows hold K/gs entries rounded up to a multiple of four."""
    for K, gs, want in [(896, 128, 8), (3584, 128, 28), (18944, 128, 148), (64, 32, 4),
                        (4096, 4096, 4), (512, 64, 8), (96, 32, 4), (160, 32, 8)]:
        assert o.w4g_scale_stride(K, gs) == want, (K, gs)


def pin_w4g_reduces_to_rowwise(o):
    """One group per row (gs = K) gives exactly the row-wise codes and scales,
    and the reference product agrees with the row-wise rescale (two fp32
    roundings) to 2^-23 relative."""
    for (M, N, K, seed) in [(2, 24, 256, 41), (1, 9, 896, 42)]:
        W = synth.normal(seed, (N, K), 0.02)
        W[3, :] = 0.0
        Wq_r, sw = o.w4_quantize(W)
        Wq_g, sg = o.w4g_quantize(W, K)
        assert np.array_equal(Wq_g, Wq_r)
        assert np.array_equal(sg[:, 0], sw) and not sg[:, 1:].any()
        X = synth.activation(seed + 7, M, K, outlier_frac=0.001)
        Y_r, Xq, sa, _ = o.w4a8_linear(X, Wq_r, sw)
        Y_g, B, Xq_g, sa_g = o.w4a8g_linear(X, Wq_g, sg, K)
        assert np.array_equal(Xq_g, Xq) and np.array_equal(sa_g, sa)
        assert np.all(np.abs(Y_r.astype(np.float64) - Y_g) <= 2.0 ** -23 * np.abs(Y_g) + 1e-300)
        assert np.all(B >= np.abs(Y_g) * (1 - 1e-15))


def pin_w4g_invariants(o):
    """Seeded N(0, 0.02) rows, gs = 128: |w - q*s_g| <= s_g/2 per element, the
    largest |w| of every group gets code +-7 with its sign, an all-zero group
    gets scale 0 and codes 0 inside a non-zero row, codes stay in [-7, 7]."""
    gs = 128
    W = synth.normal(13, (24, 896), 0.02)
    W[4, 130] *= 20.0
    W[7, 256:384] = 0.0
    Wq, sg = o.w4g_quantize(W, gs)
    G = 896 // gs
    assert sg.shape == (24, 8) and not sg[:, G:].any()
    q = decode_nibbles(Wq).astype(np.float64)
    s = np.repeat(sg[:, :G].astype(np.float64), gs, axis=1)
    err = np.abs(W.astype(np.float64) - q * s)
    assert np.all(err <= s / 2 * (1 + 2 ** -20) + 1e-45)
    assert np.all(np.abs(q) <= 7)
    for n in range(W.shape[0]):
        for g in range(G):
            grp = W[n, g * gs:(g + 1) * gs]
            if sg[n, g] == 0:
                assert not grp.any() and not q[n, g * gs:(g + 1) * gs].any()
                continue
            k = int(np.argmax(np.abs(grp)))
            assert q[n, g * gs + k] == 7 * np.sign(grp[k])
            assert sg[n, g] == f32_nearest(Fraction(float(np.max(np.abs(grp)))) / 7)
    assert sg[7, 2] == 0 and sg[7, 1] > 0


def pin_w4a8g_closed_forms(o):
    """Every code +7 with group scales 2^-g and every activation code +127:
    Y = s_a * 889 * gs * sum_g 2^-g exactly (one binary64 rounding) and B = Y;
    alternating activation signs cancel inside each group: Y = 0, B unchanged."""
    gs, G = 32, 5
    K = gs * G
    W = np.concatenate([np.full(gs, 7.0 * 2.0 ** -g) for g in range(G)]).astype(np.float32)
    W = np.stack([W, -W])
    Wq, sg = o.w4g_quantize(W, gs)
    assert np.array_equal(sg[0, :G], [2.0 ** -g for g in range(G)])
    for X, sign in [(np.ones((1, K), np.float16), 1), (np.tile(np.array([1, -1], np.float16), K // 2)[None, :], 0)]:
        Y, B, Xq, sa = o.w4a8g_linear(X, Wq, sg, gs)
        assert sa[0] == f32_nearest(Fraction(1, 127))
        mag = Fraction(float(sa[0])) * 889 * gs * sum(Fraction(1, 2 ** g) for g in range(G))
        want = float(mag) * sign
        assert Y[0, 0] == want and Y[0, 1] == -want, (Y, want)
        assert B[0, 0] == float(mag) and B[0, 1] == float(mag)


def pin_w4a8g_bruteforce(o):
    """The reference equals numpy's binary64 product of the dequantized
    operands element by element (w_k = q_k * s_g(k), x_k = q_k * s_a), and B
    equals the same sum over |products|."""
    for (M, N, K, gs, seed) in [(1, 7, 128, 32, 51), (3, 5, 256, 64, 52), (2, 6, 896, 128, 53)]:
        W = synth.normal(seed, (N, K), 0.02)
        Wq, sg = o.w4g_quantize(W, gs)
        Xq, sa = o.act_quantize(synth.activation(seed + 100, M, K))
        Y, B = o.w4a8g_ref(Xq, sa, Wq, sg, gs)
        w = decode_nibbles(Wq).astype(np.float64) * np.repeat(sg[:, :K // gs].astype(np.float64), gs, axis=1)
        x = Xq.astype(np.float64) * sa.astype(np.float64)[:, None]
        ref = x @ w.T
        mag = np.abs(x) @ np.abs(w).T
        assert np.all(np.abs(Y - ref) <= 1e-12 * mag + 1e-300)
        assert np.all(np.abs(B - mag) <= 1e-12 * mag + 1e-300)


def pin_w4a8g_error_bound(o):
    """Quantized group-wise linear vs the fp64 unquantized GEMV within the
    deterministic bound sum_k(|x| s_g/2 + |w| s_a/2 + s_g s_a/4)(1 + 2^-18),
    and closer to it than row-wise scales on the same seeded operands."""
    for (M, N, K, gs, seed) in [(1, 64, 896, 128, 61), (2, 16, 3584, 128, 62)]:
        W = synth.normal(seed, (N, K), 0.02)
        X = synth.activation(seed + 50, M, K, outlier_frac=0.001)
        Wq, sg = o.w4g_quantize(W, gs)
        Y, B, Xq, sa = o.w4a8g_linear(X, Wq, sg, gs)
        ref = X.astype(np.float64) @ W.astype(np.float64).T
        s_g = np.repeat(sg[:, :K // gs].astype(np.float64), gs, axis=1)   # [N][K]
        s_a = sa.astype(np.float64)[:, None]
        ax = np.abs(X).astype(np.float64)
        bound = ((ax @ s_g.T) / 2 + np.abs(W).astype(np.float64).sum(1)[None, :] * s_a / 2
                 + s_g.sum(1)[None, :] * s_a / 4) * (1 + 2 ** -18)
        assert np.all(np.abs(Y - ref) <= bound)
        Wq_r, sw = o.w4_quantize(W)
        Y_r = o.w4a8_linear(X, Wq_r, sw)[0].astype(np.float64)
        err_g = np.linalg.norm(Y - ref) / np.linalg.norm(ref)
        err_r = np.linalg.norm(Y_r - ref) / np.linalg.norm(ref)
        assert err_g < err_r, (err_g, err_r)


def pack_nibbles(q: np.ndarray) -> np.ndarray:
    """[N][K] codes in [-8, 7] -> [N][K/2] bytes, q[2j] in the low nibble."""
    u = (np.asarray(q, np.int64) & 0xF).astype(np.uint8)
    return (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)


def _fold_exact(acc, sg_row, gs, K, chunk=None, descending=False, fused=True):
    """The fixed binary32 order of the group-wise product for one output,
    evaluated in exact rationals with every step rounded by ``f32_nearest``
    (a single rounding for each fused multiply-add).  The keyword arguments
    give the plausible wrong orders the pins must tell apart."""
    L = chunk if chunk is not None else max(gs, 1024)
    F = Fraction(0)
    for c0 in range(0, K, L):
        groups = list(range(c0 // gs, min(c0 + L, K) // gs))
        if descending:
            groups.reverse()
        f = Fraction(0)
        for g in groups:
            a = Fraction(float(f32_nearest(Fraction(int(acc[g])))))
            p = a * Fraction(float(sg_row[g]))
            if not fused:
                p = Fraction(float(f32_nearest(p)))
            f = Fraction(float(f32_nearest(p + f)))
        F = Fraction(float(f32_nearest(F + f)))
    return F


def pin_w4a8g_f32_golden(o):
    """Hand-derived outputs of the fixed order (tests/golden/w4g_fold_order.txt):
    ascending groups, one rounding per fused step, chunks of max(gs, 1024)
    codes, the activation scale last."""
    cases = read_cases("w4g_fold_order.txt")
    assert len(cases) >= 6
    for c in cases:
        gs, K = int(c["gs"][0]), int(c["K"][0])
        ng = K // gs
        Xq = np.zeros((1, K), np.int8)
        q = np.zeros((1, K), np.int64)
        for t in c["acc"]:
            g, a = (int(v) for v in t.split(":"))
            Xq[0, g * gs], q[0, g * gs] = a, 1
        sg = np.zeros((1, o.w4g_scale_stride(K, gs)), np.float32)
        sg[0, :ng] = 1.0
        for t in c.get("s", []):
            g, v = t.split(":")
            sg[0, int(g)] = np.float32(v)
            assert Fraction(float(sg[0, int(g)])) == Fraction(v), v   # exact in binary32
        sa = np.array([np.float32(c["sa"][0])], np.float32)
        assert Fraction(float(sa[0])) == Fraction(c["sa"][0])
        Y = o.w4a8g_f32(Xq, sa, pack_nibbles(q), sg, gs)
        assert Fraction(float(Y[0, 0])) == Fraction(c["want"][0]), (c["name"], float(Y[0, 0]))
        for v in c["not"]:
            assert Fraction(v) != Fraction(c["want"][0])


def pin_w4a8g_f32_exact_rational(o):
    """Brute force on small seeded operands: every output equals the fixed
    order evaluated in exact rationals, and the operands separate that order
    from a descending fold, an unchunked fold, chunks of 512 codes and an
    unfused multiply-add (so a pin failure localises the mistake)."""
    seps = {"descending": 0, "unchunked": 0, "chunk512": 0, "unfused": 0}
    for (M, N, K, gs, seed) in [(2, 3, 2048, 32, 71), (1, 3, 3072, 128, 72), (2, 2, 2560, 64, 73),
                                (1, 3, 4096, 2048, 74), (2, 2, 1536, 512, 75)]:
        W = synth.normal(seed, (N, K), 0.02)
        Wq, sg = o.w4g_quantize(W, gs)
        Xq, sa = o.act_quantize(synth.activation(seed + 100, M, K, outlier_frac=0.002))
        Y = o.w4a8g_f32(Xq, sa, Wq, sg, gs)
        q = decode_nibbles(Wq)
        ng = K // gs
        acc = (Xq.astype(np.int64)[:, None, :] * q[None, :, :]).reshape(M, N, ng, gs).sum(-1)
        for m in range(M):
            for n in range(N):
                F = _fold_exact(acc[m, n], sg[n], gs, K)
                want = f32_nearest(F * Fraction(float(sa[m])))
                assert Y[m, n].view(np.uint32) == want.view(np.uint32), (gs, K, m, n, Y[m, n], want)
                seps["descending"] += _fold_exact(acc[m, n], sg[n], gs, K, descending=True) != F
                seps["unchunked"] += _fold_exact(acc[m, n], sg[n], gs, K, chunk=K) != F
                seps["chunk512"] += gs < 512 and _fold_exact(acc[m, n], sg[n], gs, K, chunk=512) != F
                seps["unfused"] += _fold_exact(acc[m, n], sg[n], gs, K, fused=False) != F
    assert all(v > 0 for v in seps.values()), seps


def pin_w4a8g_f32_closed_form(o):
    """Every code +7, group scales 2^-g, activations all 1 (codes 127):
    every group product and partial sum is exact, so Y is one rounding of
    889 * gs * sum_g 2^-g * s_a; alternating activation signs give +0."""
    gs, G = 64, 40
    K = gs * G
    W = np.concatenate([np.full(gs, 7.0 * 2.0 ** -(g % 8)) for g in range(G)]).astype(np.float32)
    W = np.stack([W, -W])
    Wq, sg = o.w4g_quantize(W, gs)
    X = np.ones((1, K), np.float16)
    Y, Xq, sa = o.w4a8g_linear_f32(X, Wq, sg, gs)
    exact = Fraction(889 * gs) * sum(Fraction(1, 2 ** (g % 8)) for g in range(G))
    want = f32_nearest(exact * Fraction(float(sa[0])))
    assert Y[0, 0] == want and Y[0, 1] == -want, (Y, want)
    Xa = np.tile(np.array([1, -1], np.float16), K // 2)[None, :]
    Y0, _, _ = o.w4a8g_linear_f32(Xa, Wq, sg, gs)
    assert np.all(Y0.view(np.uint32) == 0), Y0   # +0, never -0


def pin_w4a8g_f32_bound(o):
    """The fixed-order binary32 result against the binary64 reference: within
    the recursive-summation bound (groups per chunk + chunks + 1) * 2^-24 * B
    at the shapes of the benchmark (K = 3584 and 18944, gs = 128 and 32)."""
    for (M, N, K, gs, seed) in [(2, 16, 3584, 128, 81), (1, 8, 18944, 128, 82), (1, 4, 3584, 32, 83)]:
        W = synth.normal(seed, (N, K), 0.02)
        X = synth.activation(seed + 50, M, K, outlier_frac=0.001)
        Wq, sg = o.w4g_quantize(W, gs)
        Y32, Xq, sa = o.w4a8g_linear_f32(X, Wq, sg, gs)
        Y64, B = o.w4a8g_ref(Xq, sa, Wq, sg, gs)
        L = max(gs, 1024)
        n_round = L // gs + (K + L - 1) // L + 1
        assert np.all(np.abs(Y32.astype(np.float64) - Y64) <= n_round * 2.0 ** -24 * 1.001 * B + 1e-300)


# --------------------------------------------------------------------------
# s1-s3: IndexSoftmax
# --------------------------------------------------------------------------

def _decimal_lut(b, c):
    """round(255 * exp(-c i / (2^b - 1))) with 50-digit decimal arithmetic
    (c taken exactly as its binary64 value), last entry 0."""
    import decimal
    ctx = decimal.Context(prec=50)
    n = 1 << b
    out = []
    for i in range(n - 1):
        x = ctx.divide(ctx.multiply(decimal.Decimal(-c), i), n - 1)
        v = ctx.multiply(255, ctx.exp(x))
        out.append(int(v.quantize(decimal.Decimal(1), rounding=decimal.ROUND_HALF_UP)))
    return out + [0]


def pin_isx_lut(o):
    """The UINT8 exponent table against 50-digit decimal exp, for the page's
    (b, c) = (5, 6.6) and other points of its stable range."""
    assert list(o.isx_lut(5, 6.6)) == _decimal_lut(5, 6.6)
    for b, c in [(3, 5.5), (4, 7.7), (6, 6.6), (8, 5.5), (5, 4.0)]:
        assert list(o.isx_lut(b, c)) == _decimal_lut(b, c), (b, c)
    lut = o.isx_lut(5, 6.6)
    assert lut[0] == 255 and lut[31] == 0 and len(lut) == 32
    assert all(int(lut[i]) >= int(lut[i + 1]) for i in range(31))


def pin_isx_c_int(o):
    """c_int = round(c sqrt(d) / (s_Q s_K)) with halves away from zero."""
    import decimal
    assert o.isx_c_int(2.5, 1, 1.0, 1.0) == 3          # a half rounds up
    assert o.isx_c_int(3.5, 4, 1.0, 1.0) == 7          # sqrt(4) = 2 exactly
    assert o.isx_c_int(6.6, 128, 2.0 ** -5, 2.0 ** -5) == int(
        (decimal.Decimal(6.6) * decimal.Decimal(128).sqrt() * 1024).quantize(
            decimal.Decimal(1), rounding=decimal.ROUND_HALF_UP))
    s = float(np.float32(4 / 127))
    want = decimal.Decimal(6.6) * decimal.Decimal(128).sqrt() / (decimal.Decimal(s) * decimal.Decimal(s))
    assert o.isx_c_int(6.6, 128, s, s) == int(want.quantize(decimal.Decimal(1),
                                                             rounding=decimal.ROUND_HALF_UP))


def pin_isx_golden(o):
    for c in read_cases("index_softmax_closed_forms.txt"):
        row = np.array([int(v) for v in c["row"]], np.int64).astype(np.int32)[None, :]
        P = o.index_softmax(row, int(c["c_int"][0]))
        want = np.array([int(v) for v in c["p"]], np.uint8)
        assert np.array_equal(P[0], want), (c["name"], P[0], want)


def pin_isx_invariants(o):
    """Seeded int32 logits for d = 128 and per-tensor scales 4/127, spread
    like trained attention (dequantized logits with standard deviation 4):
    the row max gets the largest probability, probabilities do not increase
    with the distance from the max, every distance at or past c_int gets 0,
    the row sum is within cols/2 of 255, and P/255 keeps the direction of the
    fp64 softmax of the dequantized logits (cosine > 0.99; flatter rows lose
    more to the 8-bit probabilities, which the page names as its limit)."""
    s = float(np.float32(4 / 127))
    c_int = o.isx_c_int(6.6, 128, s, s)
    rows, cols = 16, 1000
    A = np.round(synth.normal(91, (rows, cols), 1.0) * (4.0 * math.sqrt(128) / (s * s))).astype(np.int32)
    A[3, :] = A[3, 0]                                    # a constant row: 255/1000 rounds to 0
    P = o.index_softmax(A, c_int).astype(np.int64)
    delta = A.max(1, keepdims=True).astype(np.int64) - A
    for r in range(rows):
        order = np.argsort(delta[r], kind="stable")
        assert np.all(np.diff(P[r][order]) <= 0)
        assert P[r][np.argmax(A[r])] == P[r].max()
        assert not P[r][delta[r] >= c_int].any()
        assert abs(int(P[r].sum()) - 255) <= cols // 2
    x = A.astype(np.float64) * s * s / math.sqrt(128)
    e = np.exp(x - x.max(1, keepdims=True))
    ref = e / e.sum(1, keepdims=True)
    keep = np.arange(rows) != 3
    cos = (P * ref).sum(1)[keep] / np.sqrt((P.astype(np.float64) ** 2).sum(1) * (ref ** 2).sum(1))[keep]
    assert np.all(cos > 0.99), cos
    assert not P[3].any()


# --------------------------------------------------------------------------
# b1/b2: W8A16
# --------------------------------------------------------------------------

def pin_w8_quantize(o):
    """Scale is binary16(max|w|/127) (numpy's conversion); codes satisfy
    |w - q*s| <= s/2 unless clamped at +-127; the largest |w| maps to +-127."""
    W = synth.normal(31, (40, 4096), 0.02)
    W[3] = 0
    W[7] *= 1e-3          # scale lands among binary16 subnormals: clamping matters
    W[8, 11] = 1e-5
    Wq8, sw16 = o.w8_quantize(W)
    for n in range(W.shape[0]):
        mx = np.float32(np.max(np.abs(W[n])))
        assert sw16[n] == (mx / np.float32(127.0)).astype(np.float16)
    s = sw16.astype(np.float64)[:, None]
    q = Wq8.astype(np.float64)
    w = W.astype(np.float64)
    assert np.all(np.abs(q) <= 127)
    free = np.abs(w) < 127.5 * s * (1 - 2 ** -20)
    ok = np.abs(w - q * s) <= s / 2 * (1 + 2 ** -20) + 1e-45
    assert np.all(ok | ~free)
    assert np.all(np.where(~free & (s > 0), np.abs(q) == 127, True))
    for n in range(W.shape[0]):
        if sw16[n] == 0:
            assert not Wq8[n].any()
        else:
            k = int(np.argmax(np.abs(W[n])))
            assert Wq8[n, k] == 127 * np.sign(W[n, k])


def pin_w8_sizes(o):
    """Page 2 section 3: 4096 x 27392 -> 214 MB F16, 107 MB INT8, scale 0.008 MB."""
    g = read_kv("w8a16_sizes.txt")
    K, N = int(g["K"]), int(g["N"])
    W = synth.normal(1, (2, K), 0.02)
    Wq8, sw16 = o.w8_quantize(W)
    assert Wq8.itemsize == 1 and sw16.itemsize == 2
    mib = 2.0 ** 20
    assert K * N * 2 / mib == g["f16_weight_mib"]
    assert K * N * Wq8.itemsize / mib == g["int8_weight_mib"]
    assert round(g["page_scale_count"] * sw16.itemsize / 1e6, 3) == g["page_scale_mb"] or \
        round(g["page_scale_count"] * sw16.itemsize / mib, 3) == g["page_scale_mb"]


def pin_w8a16_closed_form(o):
    """Integer weights with row max 127 have scale exactly 1: y = sum of codes * x."""
    K = 64
    W = np.zeros((3, K), np.float32)
    W[0, :] = 127
    W[1, :] = np.arange(K) - 32
    W[1, 0] = 127
    W[2, 5] = -127
    Wq8, sw16 = o.w8_quantize(W)
    assert np.all(sw16 == 1.0) and np.array_equal(Wq8.astype(np.float32), W)
    X = np.ones((1, K), np.float16)
    Y = o.w8a16_ref(X, Wq8, sw16)
    assert np.array_equal(Y[0], W.astype(np.float64).sum(1))
    X2 = np.zeros((1, K), np.float16)
    X2[0, 5] = 0.5
    assert np.array_equal(o.w8a16_ref(X2, Wq8, sw16)[0], W[:, 5].astype(np.float64) * 0.5)


def pin_w8a16_bruteforce_and_bound(o):
    """fp64 reference equals numpy's fp64 product of the dequantized matrix, is
    within sum_k |x| s/2 of the unquantized product, and cosine > 0.99 (page 2
    section 2 reports > 99% cosine similarity against F16)."""
    for (M, N, K, seed) in [(1, 32, 4096, 41), (3, 8, 1024, 42)]:
        W = synth.normal(seed, (N, K), 0.02)
        X = synth.activation(seed + 1, M, K)
        Wq8, sw16 = o.w8_quantize(W)
        Y = o.w8a16_ref(X, Wq8, sw16)
        deq = Wq8.astype(np.float64) * sw16.astype(np.float64)[:, None]
        ref = X.astype(np.float64) @ deq.T
        assert np.allclose(Y, ref, rtol=1e-12, atol=1e-12)
        exact = X.astype(np.float64) @ W.astype(np.float64).T
        bound = np.abs(X).astype(np.float64).sum(1)[:, None] * sw16.astype(np.float64)[None, :] / 2
        assert np.all(np.abs(Y - exact) <= bound * (1 + 1e-9) + 1e-12)
        cos = float((Y * exact).sum() / np.sqrt((Y ** 2).sum() * (exact ** 2).sum()))
        assert cos > 0.99



# --------------------------------------------------------------------------
# the MLP's gated product: binary64 -> binary16 and silu(g) * u
# --------------------------------------------------------------------------

def pin_double_to_half(o):
    """binary64 -> binary16 (round to nearest even) against numpy's IEEE
    conversion: random values over the whole binary16 range and beyond,
    exact ties in the normal and subnormal ranges, the overflow threshold."""
    rng = np.random.Generator(np.random.PCG64(71))
    mags = np.ldexp(rng.random(4000) + 0.5, rng.integers(-30, 18, size=4000))
    xs = np.concatenate([mags, -mags, [0.0, -0.0, 65504.0, 65519.99, 65520.0, 65536.0, 1e300, 2.0 ** -24,
                                       2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -14 - 2.0 ** -25, np.inf, -np.inf]])
    # ties: (k + 1/2) quanta for random k, normal (quantum 2^(e-10)) and subnormal (2^-24)
    k = rng.integers(1024, 2047, size=500).astype(np.float64)
    e = rng.integers(-14, 16, size=500)
    ties = np.ldexp(k + 0.5, e - 10)
    sub = np.ldexp(rng.integers(0, 1023, size=200).astype(np.float64) + 0.5, -24)
    xs = np.concatenate([xs, ties, -ties, sub, -sub])
    want = xs.astype(np.float16).view(np.uint16)
    got = np.array([o.double_to_half(x) for x in xs], np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(xs[i], hex(got[i]), hex(want[i])) for i in bad[:5]]


def _decimal_silu_mul(g, u):
    """silu(g) * u with 50-digit decimal arithmetic (independent of the
    binary64 evaluation)."""
    import decimal
    ctx = decimal.Context(prec=50)
    x = decimal.Decimal(float(g))
    return ctx.multiply(ctx.divide(x, ctx.add(1, ctx.exp(-x))), decimal.Decimal(float(u)))


def pin_silu_mul(o):
    """v = silu(g) * u against 50-digit decimal arithmetic (relative error of
    a few binary64 roundings), h = its binary16 rounding; closed forms
    (silu(0) = 0, u = 0, silu(40) = 40 in binary64, silu(-40) ~ 0) and the
    identity silu(x) - silu(-x) = x."""
    rng = np.random.Generator(np.random.PCG64(72))
    g = np.concatenate([rng.normal(0, 3, 60), [0.0, 1.0, -1.0, 40.0, -40.0, 0.5, -7.25, 12.0]]).astype(np.float32)
    u = np.concatenate([rng.normal(0, 2, 60), [5.0, 0.0, 2.0, 1.5, 3.0, -4.0, 0.125, -1.0]]).astype(np.float32)
    v, h = o.silu_mul(g, u)
    for i in range(g.size):
        ref = _decimal_silu_mul(g[i], u[i])
        rf = float(ref)
        assert abs(v[i] - rf) <= 8 * 2.0 ** -53 * abs(rf) + 1e-300, (g[i], u[i], v[i], rf)
        # h: the binary16 rounding of the exact value, unless that value sits
        # within the binary64 error of a binary16 rounding boundary
        hq = np.float64(np.float16(rf))
        lo, hi = sorted((hq, np.float64(np.nextafter(np.float16(hq), np.float16(np.sign(rf - hq) or 1)))))
        near = abs(abs(rf) - abs((lo + hi) / 2)) <= 16 * 2.0 ** -53 * abs(rf)
        if not near:
            assert h[i] == np.float16(rf).view(np.uint16), (g[i], u[i], hex(h[i]))
    assert v[g.size - 8] == 0.0 and v[g.size - 7] == 0.0       # silu(0) * 5, silu(1) * 0
    assert v[g.size - 5] == 40.0 * 1.5                          # silu(40) = 40 in binary64
    assert abs(v[g.size - 4]) < 1e-15 and h[g.size - 4] & 0x7FFF == 0
    # values just above a binary16 rounding midpoint by less than half a
    # binary32 ulp (g = 40, so silu(g) = 40 exactly and v = 40 u): rounded
    # straight from binary64 they go up; through binary32 they would land on
    # the midpoint and go to the even, lower neighbour
    found = 0
    for base in (1.0, 3.0, 100.0, 0.3, 7.0, 2000.0, 0.01, 40000.0):
        lo = np.float16(base)
        if lo.view(np.uint16) & 1:
            lo = np.nextafter(lo, np.float16(np.inf))
        hi = np.nextafter(lo, np.float16(np.inf))
        mid = (np.float64(lo) + np.float64(hi)) / 2
        half_ulp32 = np.float64(np.spacing(np.float32(mid))) / 2
        u0 = np.float32(mid / 40.0)
        for k in range(-4, 5):
            uk = np.float32(u0 + np.float32(k) * np.spacing(u0))
            v40 = 40.0 * np.float64(uk)
            if mid < v40 < mid + half_ulp32:
                vk, hk = o.silu_mul(np.array([40.0], np.float32), np.array([uk], np.float32))
                assert vk[0] == v40 and hk[0] == hi.view(np.uint16), (base, uk, hex(hk[0]))
                found += 1
    assert found >= 3, found
    x = rng.normal(0, 4, 200).astype(np.float32)
    one = np.ones_like(x)
    vp, _ = o.silu_mul(x, one)
    vm, _ = o.silu_mul(-x, one)
    assert np.all(np.abs((vp - vm) - x.astype(np.float64)) <= 8 * 2.0 ** -53 * (np.abs(x) + 1.0))


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
