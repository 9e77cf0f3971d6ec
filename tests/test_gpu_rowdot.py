"""The row-per-thread W4A8 kernel (2..8 activation rows, row-wise scales)
against the CPU oracle, bit for bit, through the C ABI: the activation codes
and scales it writes, the int32 accumulators and the fp32 outputs.  Shapes
span several 128-row tiles with ragged tails, K with a partial last 256-code
box, single-piece and split-K plans, both thread counts per weight row,
grouped launches (eager, PDL, a replayed CUDA graph), the largest sums and
the largest K.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import guards  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402

pytestmark = pytest.mark.gpu


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


@pytest.fixture(autouse=True)
def _reset_tuning(w4):
    w4.w4a8_set_tuning(qmma_max_m=1, rowdot_max_m=8)  # the row-per-thread kernel for 2..8 rows
    yield
    w4.w4a8_set_tuning(reset=True)
    assert w4.w4a8_device_error() == 0


def bits(a):
    return np.ascontiguousarray(a).view(np.uint32)


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def check(w4, orc, M, K, N, seed, fused=True, flags=0):
    plan = w4.w4a8_plan_info(M, K, N)
    assert plan["kernel"] == 2, plan
    W = synth.normal(seed, (N, K), 0.02)
    W[0] = 0  # a zero weight row: scale 0, outputs 0
    X = synth.activation(seed + 7, M, K, outlier_frac=0.001)
    X[M - 1] = 0  # a zero activation row
    Wq_ref, sw_ref = orc.w4_quantize(W)
    Y_ref, Xq_ref, sa_ref, acc_ref = orc.w4a8_linear(X, Wq_ref, sw_ref)
    Wq, sw = w4.w4_quantize_weights(to_dev(W))
    gacc, gY = guards.out((M, N), torch.int32), guards.out((M, N), torch.float32)
    gXq, gsa = guards.out((M, K), torch.int8), guards.out((M,), torch.float32)
    gws = guards.workspace(w4.w4a8_workspace_bytes(M, K, N))
    Xq, sa, acc = gXq.t, gsa.t, gacc.t
    if fused:
        Y = w4.w4a8_linear(to_dev(X), Wq, sw, Y=gY.t, Xq_out=Xq, sa_out=sa, acc_out=acc,
                           ws=guards.t(gws), flags=flags)
    else:
        w4.act_quantize_i8(to_dev(X), Xq=Xq, sa=sa)
        Y = w4.w4a8_gemv(Xq, sa, Wq, sw, Y=gY.t, acc_out=acc, ws=guards.t(gws), flags=flags)
    guards.check_all(gacc, gY, gXq, gsa, gws)
    assert np.array_equal(Xq.cpu().numpy(), Xq_ref)
    assert np.array_equal(bits(sa.cpu().numpy()), bits(sa_ref))
    assert np.array_equal(acc.cpu().numpy(), acc_ref)
    assert np.array_equal(bits(Y.cpu().numpy()), bits(Y_ref))
    return plan


ROWDOT_SHAPES = [
    (2, 3584, 1000, 0),      # split K (8 tiles)
    (3, 896, 129, 1),        # one row past a tile
    (4, 18944, 300, 2),      # long rows, many pieces
    (5, 288, 77, 3),         # a 32-code tail box
    (6, 32, 5, 4),           # the smallest K: one partial box
    (7, 3584, 40000, 5),     # more tiles than CTA slots: one piece per tile
    (8, 3584, 18944, 6),     # gate projection
    (8, 18944, 3584, 7),     # down projection
    (2, 131072, 3, 8),       # the largest K
]


@pytest.mark.parametrize("tpr", [0, 2, 8])
@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("M,K,N,seed", ROWDOT_SHAPES)
def test_rowdot_parity(w4, orc, M, K, N, seed, fused, tpr):
    if tpr:
        w4.w4a8_set_tuning(force_threads_per_row=tpr, qmma_max_m=1, rowdot_max_m=8)
    plan = check(w4, orc, M, K, N, seed, fused=fused)
    assert plan["threads_per_row"] == (tpr or 4)


def test_rowdot_plans_cover_split_and_whole(w4):
    """The shapes above reach both one-piece and split-K plans."""
    assert w4.w4a8_plan_info(7, 3584, 40000)["splits"] == 1
    assert w4.w4a8_plan_info(4, 18944, 300)["splits"] > 1
    assert w4.w4a8_plan_info(2, 131072, 3)["splits"] > 1


def test_rowdot_tickets_reset_and_pdl(w4, orc):
    """Back-to-back split-K calls sharing one workspace (tickets handed back
    by the last CTA of each tile), with and without programmatic launch."""
    for rep in range(3):
        check(w4, orc, 4, 3584, 700, 20 + rep, flags=w4.LAUNCH_PDL if rep else 0)


def test_rowdot_largest_sums(w4):
    """Every weight code -8 against activation codes +127 / -127: each row's
    sum is -+1016 K, each thread's partial 16 x that over its share, the
    largest magnitudes the int32 accumulators meet."""
    K, N = 131072, 130
    for M in (2, 8):
        Wq = torch.full((N, K // 2), 0x88, dtype=torch.uint8, device="cuda")
        sw = torch.ones((N,), dtype=torch.float32, device="cuda")
        Xq = torch.full((M, K), 127, dtype=torch.int8, device="cuda")
        Xq[1::2] = -127
        sa = torch.ones((M,), dtype=torch.float32, device="cuda")
        acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
        Y = w4.w4a8_gemv(Xq, sa, Wq, sw, acc_out=acc)
        torch.cuda.synchronize()
        want = np.where(np.arange(M)[:, None] % 2 == 0, -1016 * K, 1016 * K) * np.ones((1, N), np.int64)
        assert np.array_equal(acc.cpu().numpy(), want)
        assert np.array_equal(Y.cpu().numpy(), want.astype(np.float32))


def test_rowdot_every_code_pair(w4):
    """All 16 weight codes against all 255 activation codes: one weight row
    per code, activations -127..127 laid along K; each sum has a closed
    form q * sum(a) over the row, and the single-code rows check the nibble
    order (even codes in the low nibble)."""
    M, K = 2, 256
    codes = np.arange(-8, 8)
    N = len(codes) + 2
    Wq = np.zeros((N, K // 2), np.uint8)
    for i, q in enumerate(codes):
        Wq[i] = (q & 0xF) | ((q & 0xF) << 4)
    Wq[16, 0] = 0x07      # code 7 at position 0 only
    Wq[17, 0] = 0x70      # code 7 at position 1 only
    a = np.zeros((M, K), np.int8)
    a[0, :255] = np.arange(-127, 128)
    a[1, :255] = np.arange(127, -128, -1)
    a[1, 0], a[1, 1] = 5, -3
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    w4.w4a8_gemv(to_dev(a), to_dev(np.ones(M, np.float32)), to_dev(Wq),
                 to_dev(np.ones(N, np.float32)), acc_out=acc)
    torch.cuda.synchronize()
    got = acc.cpu().numpy()
    s = a.astype(np.int64).sum(axis=1)
    for i, q in enumerate(codes):
        assert np.array_equal(got[:, i], q * s)
    assert list(got[:, 16]) == [7 * -127, 7 * 5]
    assert list(got[:, 17]) == [7 * -126, 7 * -3]


@pytest.mark.parametrize("M", [2, 5, 8])
def test_rowdot_grouped_and_graph(w4, orc, M):
    """gate/up-style grouped launches (one plan per matrix, one activation
    pass), eager, with PDL, and replayed from a CUDA graph."""
    K, Ns = 3584, (1000, 129, 7)
    X = synth.activation(700 + M, M, K, outlier_frac=0.001)
    Wqs, sws, refs = [], [], []
    for g, N in enumerate(Ns):
        W = synth.normal(710 + g, (N, K), 0.02)
        Wq_ref, sw_ref = orc.w4_quantize(W)
        refs.append(orc.w4a8_linear(X, Wq_ref, sw_ref)[0])
        Wq, sw = w4.w4_quantize_weights(to_dev(W))
        Wqs.append(Wq)
        sws.append(sw)
    Xd = to_dev(X)
    for rep in range(2):
        Ys = w4.w4a8_linear_grouped(Xd, Wqs, sws, flags=w4.LAUNCH_PDL if rep else 0)
        torch.cuda.synchronize()
        for Y, ref in zip(Ys, refs):
            assert np.array_equal(bits(Y.cpu().numpy()), bits(ref))
    Ys = [torch.empty((M, N), dtype=torch.float32, device="cuda") for N in Ns]
    ws = torch.zeros((w4.w4a8_workspace_bytes(M, K, sum(Ns)),), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        w4.w4a8_linear_grouped(Xd, Wqs, sws, Ys=Ys, ws=ws, flags=w4.LAUNCH_PDL)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        w4.w4a8_linear_grouped(Xd, Wqs, sws, Ys=Ys, ws=ws, flags=w4.LAUNCH_PDL)
    for _ in range(2):
        for Y in Ys:
            Y.zero_()
        g.replay()
        torch.cuda.synchronize()
        for Y, ref in zip(Ys, refs):
            assert np.array_equal(bits(Y.cpu().numpy()), bits(ref))


def test_rowdot_matches_other_kernels(w4):
    """The same call on the row-per-thread kernel, the tensor cores and the
    dp4a GEMV gives the same bits."""
    M, K, N = 6, 3584, 1000
    W = synth.normal(730, (N, K), 0.02)
    X = to_dev(synth.activation(731, M, K, outlier_frac=0.001))
    Wq, sw = w4.w4_quantize_weights(to_dev(W))
    outs = []
    for kw in (dict(rowdot_max_m=8), dict(rowdot_max_m=1), dict(rowdot_max_m=1, mma_min_m=65)):
        w4.w4a8_set_tuning(qmma_max_m=1, **kw)
        outs.append(w4.w4a8_linear(X, Wq, sw).cpu().numpy())
    assert np.array_equal(bits(outs[0]), bits(outs[1]))
    assert np.array_equal(bits(outs[0]), bits(outs[2]))
