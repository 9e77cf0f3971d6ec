"""The MLP's gated product h = binary16(silu(g) * u) between the gate/up and
down projections, against the CPU oracle.

Contract (include/w4a8.h): g and u (the gate/up outputs) are bit-exact; h
equals the oracle's binary16 rounding of v = silu(g) * u (binary64), except
where v lies within 2^-20 |v| of a binary16 rounding boundary, where the
other neighbour is allowed too; such cases are counted.  The down projection
of h is then bit-exact against the oracle on the same h.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import guards  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402

pytestmark = pytest.mark.gpu

REL = 2.0 ** -20  # the contract's distance to a rounding boundary


@pytest.fixture(scope="module")
def w4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_weight_quantized_w4a8_gb300 as m
    m.build()
    m.w4a8_set_tuning(reset=True)
    return m


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


@pytest.fixture(autouse=True)
def _reset_tuning(w4):
    w4.w4a8_set_tuning(reset=True)
    yield
    w4.w4a8_set_tuning(reset=True)
    assert w4.w4a8_device_error() == 0


def bits(a):
    a = np.ascontiguousarray(a)
    return a.view(np.uint32 if a.dtype.itemsize == 4 else np.uint16)


def check_h(h_gpu, v, h_ref):
    """h_gpu (uint16 bits) against the oracle: equal, or the two adjacent
    binary16 neighbours of a v within REL |v| of their midpoint.  Returns the
    number of such boundary cases."""
    h_gpu = np.ascontiguousarray(h_gpu).reshape(-1)
    v = np.ascontiguousarray(v).reshape(-1)
    h_ref = np.ascontiguousarray(h_ref).reshape(-1)
    bad = np.nonzero(h_gpu != h_ref)[0]
    for i in bad:
        a = np.float64(h_gpu[i:i + 1].view(np.float16)[0])
        b = np.float64(h_ref[i:i + 1].view(np.float16)[0])
        lo, hi = min(a, b), max(a, b)
        assert np.float16(lo) != np.float16(hi) and np.nextafter(np.float16(lo), np.float16(np.inf)) == np.float16(hi), \
            ("not neighbours", i, v[i], hex(h_gpu[i]), hex(h_ref[i]))
        assert abs(v[i] - (lo + hi) / 2) <= REL * abs(v[i]), ("not at a boundary", i, v[i], a, b)
    return bad.size


def gate_up_weights(w4, orc, N, K, seed):
    Wg = synth.normal_host(seed, (N, K), 0.02)
    Wu = synth.normal_host(seed + 1, (N, K), 0.02)
    refs = [orc.w4_quantize(Wg), orc.w4_quantize(Wu)]
    (Wqg, swg), (Wqu, swu) = w4.w4_quantize_weights(torch.from_numpy(Wg).cuda()), \
        w4.w4_quantize_weights(torch.from_numpy(Wu).cuda())
    Wq_gu, sw_gu = w4.w4_interleave_rows(Wqg, swg, Wqu, swu)
    inter = np.empty((2 * N, K // 2), np.uint8)
    inter[0::2], inter[1::2] = refs[0][0], refs[1][0]
    assert np.array_equal(Wq_gu.cpu().numpy(), inter)
    sint = np.empty(2 * N, np.float32)
    sint[0::2], sint[1::2] = refs[0][1], refs[1][1]
    assert np.array_equal(bits(sw_gu.cpu().numpy()), bits(sint))
    return Wq_gu, sw_gu, refs


def run_gate_up_silu(w4, orc, M, K, N, seed, flags=0):
    Wq_gu, sw_gu, refs = gate_up_weights(w4, orc, N, K, seed)
    X = synth.activation(seed + 500, M, K, outlier_frac=0.001)
    gH, gY = guards.out((M, N), torch.float16), guards.out((M, 2 * N), torch.float32)
    gws = guards.workspace(w4.w4a8_gate_up_silu_workspace_bytes(M, K, N))
    H, Y = w4.w4a8_gate_up_silu(torch.from_numpy(X).cuda(), Wq_gu, sw_gu, H=gH.t, Y_gu=gY.t,
                                ws=guards.t(gws), flags=flags)
    guards.check_all(gH, gY, gws)
    g_ref = orc.w4a8_linear(X, *refs[0])[0]
    u_ref = orc.w4a8_linear(X, *refs[1])[0]
    Yh = Y.cpu().numpy()
    assert np.array_equal(bits(Yh[:, 0::2]), bits(g_ref)), "gate outputs differ"
    assert np.array_equal(bits(Yh[:, 1::2]), bits(u_ref)), "up outputs differ"
    v, h_ref = orc.silu_mul(g_ref, u_ref)
    n_boundary = check_h(H.cpu().numpy().view(np.uint16), v, h_ref)
    return H, h_ref, n_boundary


@pytest.mark.parametrize("M,K,N,seed,splits", [(1, 3584, 300, 1400, 0), (1, 896, 1001, 1402, 0),
                                               (1, 3584, 700, 1404, 3), (1, 18944, 64, 1406, 0),
                                               (2, 1024, 260, 1408, 0), (5, 3584, 129, 1410, 0),
                                               (16, 512, 77, 1412, 0), (40, 288, 33, 1414, 0)])
def test_gate_up_silu_shapes(w4, orc, M, K, N, seed, splits):
    """One row (the fused epilogue; split K through the last CTA) and batches
    (the linear on the interleaved matrix, then the product's own kernel);
    an odd number of pairs, ragged tiles."""
    if splits:
        w4.w4a8_set_tuning(force_splits=splits)
    _, _, nb = run_gate_up_silu(w4, orc, M, K, N, seed)
    assert nb <= max(2, M * N // 1000)


def test_gate_up_silu_then_down_full_size(w4, orc):
    """The Qwen2-7B-shaped MLP at one row: gate/up 3584 -> 18944 with the
    product in the epilogue, then down 18944 -> 3584 on h; every output."""
    K, N = 3584, 18944
    H, h_ref, nb = run_gate_up_silu(w4, orc, 1, K, N, 1004, flags=w4.LAUNCH_PDL)
    assert nb <= 20
    Wd = synth.normal_host(1006, (K, N), 0.02)
    Wqd_ref, swd_ref = orc.w4_quantize(Wd)
    Wqd, swd = w4.w4_quantize_weights(torch.from_numpy(Wd).cuda())
    h16 = h_ref.view(np.float16).reshape(1, N)
    Y_ref = orc.w4a8_linear(h16, Wqd_ref, swd_ref)[0]
    # down on the oracle's h, and (when the two agree everywhere) on the GPU's
    Yd = w4.w4a8_linear(torch.from_numpy(h16).cuda(), Wqd, swd, flags=w4.LAUNCH_PDL)
    assert np.array_equal(bits(Yd.cpu().numpy()), bits(Y_ref))
    if nb == 0:
        Yd2 = w4.w4a8_linear(H, Wqd, swd, flags=w4.LAUNCH_PDL)
        assert np.array_equal(bits(Yd2.cpu().numpy()), bits(Y_ref))


def test_silu_mul_standalone(w4, orc):
    """The product's own kernel on fp32 inputs over the whole range that
    matters: large |g| (silu -> g or -> 0), zeros, signs, tiny products
    (binary16 subnormals) and overflow past 65504."""
    rng = np.random.Generator(np.random.PCG64(1420))
    M, N = 3, 5000
    g = (rng.standard_normal((M, N)) * rng.choice([0.01, 1, 8, 60], size=(M, N))).astype(np.float32)
    u = (rng.standard_normal((M, N)) * rng.choice([1e-6, 1, 100, 5000], size=(M, N))).astype(np.float32)
    g[0, :4] = [0.0, -0.0, 100.0, -100.0]
    u[0, 4:8] = 0.0
    v, h_ref = orc.silu_mul(g, u)
    gH = guards.out((M, N), torch.float16)
    H = w4.w4a8_silu_mul(torch.from_numpy(g).cuda(), torch.from_numpy(u).cuda(), H=gH.t)
    guards.check_all(gH)
    nb = check_h(H.cpu().numpy().view(np.uint16), v, h_ref)
    assert nb <= 10
