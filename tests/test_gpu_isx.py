"""IndexSoftmax: CUDA path vs the CPU oracle through the C ABI, bit for bit.

Every kernel path is exercised: the vector register path (cols % 4 == 0,
1 to 8 accesses of four logits per thread), the scalar register path (other
cols) and the streaming path (rows longer than the registers hold); table
indices exactly at, just below and just above every rounding threshold;
the int32 extremes; c_int = 0 and c_int = 2^31 - 1; table sizes b = 1..8.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import guards  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402

pytestmark = pytest.mark.gpu

S_QK = float(np.float32(4 / 127))  # per-tensor INT8 scale of N(0, 1) data clipped at 4 sigma


@pytest.fixture(scope="module")
def w4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_weight_quantized_w4a8_gb300 as m
    m.build()
    m.lib()
    return m


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def logits(seed, rows, cols, std_real=4.0, d=128):
    """int32 logits whose dequantized values (x s_q s_k / sqrt(d)) have
    standard deviation std_real."""
    z = synth.normal(seed, (rows, cols), 1.0).astype(np.float64)
    return np.round(z * std_real * math.sqrt(d) / (S_QK * S_QK)).astype(np.int32)


def check(w4, orc, A, c_int, b=5, lut=None):
    P_ref = orc.index_softmax(A, c_int, b, lut)
    Ad = torch.from_numpy(np.ascontiguousarray(A)).cuda()
    gP = guards.out(A.shape, torch.uint8)
    P = w4.index_softmax_u8(Ad, c_int, b, None if lut is None else bytes(lut), P=gP.t)
    guards.check_all(gP)
    got = P.cpu().numpy()
    bad = np.argwhere(got != P_ref)
    assert bad.size == 0, (bad[:5], got[tuple(bad[0])], P_ref[tuple(bad[0])])
    return got


def test_isx_golden(w4, orc):
    from pins import read_cases
    for c in read_cases("index_softmax_closed_forms.txt"):
        row = np.array([int(v) for v in c["row"]], np.int64).astype(np.int32)[None, :]
        got = check(w4, orc, row, int(c["c_int"][0]))
        assert list(got[0]) == [int(v) for v in c["p"]], c["name"]


@pytest.mark.parametrize("rows,cols", [(1, 1), (3, 3), (5, 4), (7, 17), (2, 64), (9, 1000),
                                       (4, 1024), (3, 2048), (5, 4095), (6, 4096), (2, 8192),
                                       (3, 8196), (2, 2051), (2, 20000), (1, 65537)])
def test_isx_shapes(w4, orc, rows, cols):
    c_int = orc.isx_c_int(6.6, 128, S_QK, S_QK)
    A = logits(100 + cols, rows, cols)
    check(w4, orc, A, c_int)


@pytest.mark.parametrize("std_real", [0.5, 1.0, 4.0, 16.0])
def test_isx_spreads(w4, orc, std_real):
    c_int = orc.isx_c_int(6.6, 128, S_QK, S_QK)
    check(w4, orc, logits(7, 33, 4096, std_real), c_int)


def test_isx_thresholds_exact(w4, orc):
    """Distances exactly at, one below and one above every rounding
    threshold of every index, for thresholds that are and are not integers."""
    for c_int in (62, 63, 1000, 31, 75273, 2 ** 31 - 1, 1, 2, 3):
        top = 31
        deltas = set()
        for k in range(1, top + 1):
            t = -(-c_int * (2 * k - 1) // (2 * top))
            deltas.update({t - 1, t, t + 1})
        deltas = sorted(d for d in deltas if 0 <= d <= 2 ** 31 - 1)
        # one row per group of distances, the row max first
        cols = 64
        rows = []
        for i in range(0, len(deltas), cols - 1):
            chunk = deltas[i:i + cols - 1]
            base = 2 ** 31 - 1
            row = [base] + [base - d for d in chunk]
            row += [base] * (cols - len(row))
            rows.append(row)
        A = np.array(rows, np.int64).astype(np.int32)
        check(w4, orc, A, c_int)


@pytest.mark.parametrize("b", [1, 2, 3, 5, 6, 8])
def test_isx_table_sizes(w4, orc, b):
    c_int = orc.isx_c_int(6.6, 128, S_QK, S_QK)
    lut = orc.isx_lut(b, 6.6)
    if lut[0] == 0:
        pytest.skip("table without a positive first entry")
    check(w4, orc, logits(11, 17, 1000), c_int, b, lut)


def test_isx_extremes(w4, orc):
    A = np.array([[2 ** 31 - 1, -2 ** 31, 0, 5] * 4,
                  [-2 ** 31] * 16,
                  [2 ** 31 - 1] * 16,
                  list(range(-8, 8))], np.int64).astype(np.int32)
    for c_int in (0, 1, 7, 2 ** 31 - 1):
        check(w4, orc, A, c_int)


def test_isx_custom_table(w4, orc):
    lut = np.array([200, 150, 150, 1] + [0] * 28, np.uint8)
    check(w4, orc, logits(13, 9, 333), 5000, 5, lut)


def test_isx_attention_shape_sampled(w4, orc):
    """The benchmark's shape, 32 heads x 1024 query rows x 4096 keys
    (512 MB of logits), checked on sampled rows."""
    rows, cols = 32 * 1024, 4096
    c_int = orc.isx_c_int(6.6, 128, S_QK, S_QK)
    A = torch.empty((rows, cols), dtype=torch.int32, device="cuda")
    chunk = 2048
    for r0 in range(0, rows, chunk):
        z = synth.normal_gpu(4242, (chunk, cols), 1.0, offset=r0 * cols)
        A[r0:r0 + chunk] = torch.round(z.double() * (4.0 * math.sqrt(128) / (S_QK * S_QK))).int()
    P = w4.index_softmax_u8(A, c_int)
    torch.cuda.synchronize()
    rng = np.random.Generator(np.random.PCG64(5))
    sample = np.array(sorted(set(rng.choice(rows, 48, replace=False).tolist()) | {0, rows - 1}))
    idx = torch.from_numpy(sample).cuda()
    # the sampled rows regenerated on the host by the generator's CPU twin
    scale = 4.0 * math.sqrt(128) / (S_QK * S_QK)
    A_rows = np.stack([np.round(synth.normal(4242, (cols,), 1.0, offset=int(r) * cols)
                                .astype(np.float64) * scale).astype(np.int32) for r in sample])
    assert np.array_equal(A[idx].cpu().numpy(), A_rows)
    P_ref = orc.index_softmax(A_rows, c_int)
    assert np.array_equal(P[idx].cpu().numpy(), P_ref)


def test_isx_longest_rows(w4, orc):
    """Rows of ISX_MAX_COLS = 2^23 logits (streaming path): a seeded row, and a
    row of equal logits whose sum reaches 255 * 2^23, the largest the int32
    row sum has to hold."""
    cols = 1 << 23
    c_int = orc.isx_c_int(6.6, 128, S_QK, S_QK)
    A = np.concatenate([logits(120, 1, cols), np.full((1, cols), -5, np.int32)])
    P = check(w4, orc, A, c_int)
    assert not P[1].any()  # 255 * 255 / (255 * 2^23) rounds to 0
