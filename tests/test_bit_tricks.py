"""Exhaustive host checks of the bit-level identities the kernels rely on,
emulated with numpy (no GPU): every INT4 nibble value in every position of a
packed word, and every INT8 activation code."""
import numpy as np


def f16(bits):
    return float(np.array([bits], dtype=np.uint16).view(np.float16)[0])


def code(n):
    return n - 16 if n >= 8 else n


def test_binary16_nibble_widening():
    """Tensor-core converters: (w & 0x000F000F) ^ 0x64086408 is 1032 + q for
    nibbles 0 and 4, (w & 0x00F000F0) ^ 0x64806480 is 1024 + 16 (q + 8) for
    nibbles 1 and 5 (then * 1/16 - 72), and the word shifted by 8 gives
    nibbles 2, 6 and 3, 7; pair t holds codes (t, t + 4)."""
    for n in range(16):
        for pos in range(8):
            w = n << (4 * pos)
            w2 = w >> 8
            words = [((w & 0x000F000F) ^ 0x64086408, 0), ((w & 0x00F000F0) ^ 0x64806480, 1),
                     ((w2 & 0x000F000F) ^ 0x64086408, 0), ((w2 & 0x00F000F0) ^ 0x64806480, 1)]
            for t, (x, scaled) in enumerate(words):
                for half in (0, 1):
                    h = f16((x >> (16 * half)) & 0xFFFF)
                    v = h * 0.0625 - 72.0 if scaled else h - 1032.0
                    want = code(n) if t + 4 * half == pos else 0
                    assert v == want, (n, pos, t, half, v)


def test_rowdot_signed_nibbles_times_16():
    """Row-per-thread kernel: (w << 4) & 0xF0F0F0F0 and w & 0xF0F0F0F0 hold
    16 q of the even and odd codes as signed bytes, so a signed dp4a against
    the activation codes gives 16 x the products exactly."""
    rng = np.random.Generator(np.random.PCG64(5))
    for n in range(16):
        for pos in range(8):
            w = n << (4 * pos)
            lo = (w << 4) & 0xF0F0F0F0
            hi = w & 0xF0F0F0F0
            for b in range(4):
                sl = np.int8(np.uint8((lo >> (8 * b)) & 0xFF))
                sh = np.int8(np.uint8((hi >> (8 * b)) & 0xFF))
                assert int(sl) == (16 * code(n) if pos == 2 * b else 0)
                assert int(sh) == (16 * code(n) if pos == 2 * b + 1 else 0)
    # random words against random codes: the dp4a sums equal 16 x the dot
    for _ in range(200):
        w = int(rng.integers(0, 2 ** 32))
        a = rng.integers(-127, 128, size=8)
        q = np.array([code((w >> (4 * k)) & 0xF) for k in range(8)])
        lo = (w << 4) & 0xF0F0F0F0
        hi = w & 0xF0F0F0F0
        s = 0
        for b in range(4):
            s += int(np.int8(np.uint8((lo >> (8 * b)) & 0xFF))) * int(a[2 * b])
            s += int(np.int8(np.uint8((hi >> (8 * b)) & 0xFF))) * int(a[2 * b + 1])
        assert s == 16 * int(np.dot(q, a)) and s % 16 == 0


def test_e4m3_activation_split():
    """e4m3 tensor-core path: a = 16 (a >> 4) + (a & 15) with a >> 4 in
    [-8, 7] and a & 15 in [0, 15]: integers of magnitude at most 16, exact
    in e4m3 (3 mantissa bits plus the implicit one)."""
    for a in range(-127, 128):
        hi, lo = a >> 4, a & 15
        assert 16 * hi + lo == a and -8 <= hi <= 7 and 0 <= lo <= 15
        # every integer of magnitude <= 16 is exact in e4m3
        assert abs(hi) <= 16 and abs(lo) <= 16
