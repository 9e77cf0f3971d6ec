"""The warp-level MMA kernel (2..32 batch rows) against the CPU oracle,
element by element, through the C ABI, with both operand types.

binary16: every INT4 weight code and INT8 activation code is an exact
binary16 integer (m16n8k16).  e4m3: weight codes become the bytes v = q + 8
(exactly v * 2^-9) and activation codes two exact e4m3 integers
(a = 16 a_hi + a_lo, m16n8k32).  Either way the fp32 sums of the MMAs are
exact, so the int32 accumulators, Xq, s_a and Y must equal the oracle's bit
for bit.  Shapes span one and several 128-row tiles, ragged row and K tails
(a partial last 256-code box), split K, every n-tile count and the largest
sums.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import guards  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402

pytestmark = pytest.mark.gpu

QMMA = 3  # w4a8_plan_info "kernel" of the warp-level MMA kernel


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


@pytest.fixture(params=[1, 2], ids=["binary16", "e4m3"])
def ops(request):
    """Operand type of the kernel (w4a8_tuning_t.qmma_operands)."""
    return request.param


@pytest.fixture(autouse=True)
def _reset_tuning(w4, ops):
    w4.w4a8_set_tuning(qmma_max_m=32, qmma_operands=ops)  # every matrix, 2..32 rows
    yield
    w4.w4a8_set_tuning(reset=True)
    assert w4.w4a8_device_error() == 0


def bits(a):
    return np.ascontiguousarray(a).view(np.uint32)


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def check(w4, orc, M, K, N, seed, fused=True, flags=0):
    plan = w4.w4a8_plan_info(M, K, N)
    assert plan["kernel"] == QMMA, plan
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


QMMA_SHAPES = [
    (2, 3584, 1000, 0),      # split K (8 tiles), one n-tile
    (3, 896, 129, 1),        # one row past a tile
    (4, 18944, 300, 2),      # long rows, many pieces
    (5, 96, 77, 3),          # one partial box, two n-tiles
    (8, 3584, 256, 4),       # exactly two tiles
    (9, 1024, 1500, 5),      # three n-tiles
    (12, 2048, 640, 6),
    (16, 18944, 200, 7),     # four tiles per warp, split K
    (17, 3584, 129, 8),      # five n-tiles
    (24, 512, 4000, 9),
    (31, 288, 7, 10),        # a partial last box, seven rows
    (32, 3584, 1100, 11),    # eight n-tiles
]


@pytest.mark.parametrize("M,K,N,seed", QMMA_SHAPES)
@pytest.mark.parametrize("fused", [True, False])
def test_qmma_parity(w4, orc, M, K, N, seed, fused):
    check(w4, orc, M, K, N, 900 + seed, fused=fused)


@pytest.mark.parametrize("M,K,N,seed", [
    (2, 1024, 40000, 40),    # 313 tiles: one or two per CTA (two CTAs per SM), ragged last tile
    (7, 3584, 19457, 41),    # one tile more than 152 SMs, the last of one row
    (9, 1024, 20000, 45),    # three n-tiles: one CTA per SM
    (16, 512, 30000, 42),    # two boxes per tile
    (20, 288, 20000, 43),    # one partial box per tile, two tiles per warp
    (32, 1024, 25600, 44),   # eight n-tiles
])
def test_qmma_persistent_tiles(w4, orc, ops, M, K, N, seed):
    """One K piece and more tiles than SMs: each CTA walks tiles b, b + grid,
    ... with one ring across tile boundaries; every output bit for bit."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p = w4.w4a8_plan_info(M, K, N)
    tiles = p["ctas_per_split"]
    assert p["splits"] == 1 and tiles > sms
    two = M <= (16 if ops == 1 else 8)  # two CTAs per SM up to two n-tiles
    assert p["grid"] == (min(tiles, 2 * sms) if two else sms)
    check(w4, orc, M, K, N, 900 + seed)
    check(w4, orc, M, K, N, 900 + seed, fused=False, flags=w4.LAUNCH_PDL)


@pytest.mark.parametrize("M", [2, 6, 32])
def test_qmma_longest_rows(w4, orc, M):
    """K = 131072: every warp sums the most codes its fp32 sums hold exactly
    (16384 binary16 products, 65536 e4m3 ones), the pieces meet in int32."""
    p = check(w4, orc, M, 131072, 5, 950 + M)
    assert p["splits"] >= 2


@pytest.mark.parametrize("M", [4, 32])
@pytest.mark.parametrize("K", [4096, 131072])
def test_qmma_largest_sums(w4, M, K):
    """Weight codes 7 and -8 (nibble 0x8, legal on input) against activation
    codes +127 and -127: the largest products (binary16 |q a| = 1016; e4m3
    bytes v = 15 and v = 0) and the e4m3 bias correction 8 * sum(a) at its
    extremes."""
    N = 256
    Wq = torch.full((N, K // 2), 0x77, dtype=torch.uint8, device="cuda")
    Wq[1::2] = 0x88                            # odd rows: every code -8
    sw = torch.ones((N,), dtype=torch.float32, device="cuda")
    Xq = torch.full((M, K), 127, dtype=torch.int8, device="cuda")
    Xq[1::2] = -127
    sa = torch.ones((M,), dtype=torch.float32, device="cuda")
    assert w4.w4a8_plan_info(M, K, N)["kernel"] == QMMA
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    Y = w4.w4a8_gemv(Xq, sa, Wq, sw, acc_out=acc)
    torch.cuda.synchronize()
    a = np.where(np.arange(M) % 2 == 0, 127, -127).astype(np.int64)[:, None]
    q = np.where(np.arange(N) % 2 == 0, 7, -8).astype(np.int64)[None, :]
    want = a * q * K
    assert np.array_equal(acc.cpu().numpy(), want)
    assert np.array_equal(Y.cpu().numpy(), want.astype(np.float32))


def test_qmma_grouped(w4, orc):
    M, K, Ns = 10, 1024, (300, 7, 129)
    X = synth.activation(960, M, K, outlier_frac=0.001)
    Wqs, sws, refs = [], [], []
    for g, N in enumerate(Ns):
        W = synth.normal(961 + g, (N, K), 0.02)
        Wq_ref, sw_ref = orc.w4_quantize(W)
        refs.append(orc.w4a8_linear(X, Wq_ref, sw_ref)[0])
        Wq, sw = w4.w4_quantize_weights(to_dev(W))
        Wqs.append(Wq)
        sws.append(sw)
    assert w4.w4a8_plan_info(M, K, sum(Ns))["kernel"] == QMMA
    for rep in range(2):
        gYs = [guards.out((M, N), torch.float32) for N in Ns]
        gws = guards.workspace(w4.w4a8_workspace_bytes(M, K, sum(Ns)))
        Ys = w4.w4a8_linear_grouped(to_dev(X), Wqs, sws, Ys=[g.t for g in gYs], ws=guards.t(gws),
                                    flags=w4.LAUNCH_PDL if rep else 0)
        guards.check_all(gws, *gYs)
        for Y, ref in zip(Ys, refs):
            assert np.array_equal(bits(Y.cpu().numpy()), bits(ref))


def test_qmma_matches_other_kernels(w4, ops):
    """The same call on the warp-level MMA kernel, the row-per-thread kernel,
    the tensor cores and the dp4a GEMV gives the same bits."""
    M, K, N = 6, 3584, 1000
    W = synth.normal(970, (N, K), 0.02)
    X = to_dev(synth.activation(971, M, K, outlier_frac=0.001))
    Wq, sw = w4.w4_quantize_weights(to_dev(W))
    outs = []
    for kw, kind in ((dict(qmma_max_m=8, qmma_operands=ops), QMMA), (dict(qmma_max_m=1, rowdot_max_m=8), 2), (dict(qmma_max_m=1, rowdot_max_m=1), 1),
                     (dict(qmma_max_m=1, rowdot_max_m=1, mma_min_m=65), 0)):
        w4.w4a8_set_tuning(**kw)
        assert w4.w4a8_plan_info(M, K, N)["kernel"] == kind
        outs.append(w4.w4a8_linear(X, Wq, sw).cpu().numpy())
    for o in outs[1:]:
        assert np.array_equal(bits(outs[0]), bits(o))


def test_qmma_pdl_chain_and_graph(w4, orc):
    """Programmatically dependent launches back to back on one workspace,
    then the same chain replayed from a CUDA graph: identical bits."""
    M, K, N = 8, 3584, 700
    W = synth.normal(980, (N, K), 0.02)
    Wq_ref, sw_ref = orc.w4_quantize(W)
    Wq, sw = w4.w4_quantize_weights(to_dev(W))
    Xs = [synth.activation(981 + i, M, K, outlier_frac=0.001) for i in range(3)]
    refs = [orc.w4a8_linear(X, Wq_ref, sw_ref)[0] for X in Xs]
    Xd = [to_dev(X) for X in Xs]
    Ys = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _ in Xs]
    ws = torch.zeros(w4.w4a8_workspace_bytes(M, K, N), dtype=torch.uint8, device="cuda")

    def chain():
        for X, Y in zip(Xd, Ys):
            w4.w4a8_linear(X, Wq, sw, Y=Y, ws=ws, flags=w4.LAUNCH_PDL)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        chain()
    torch.cuda.synchronize()
    for Y, ref in zip(Ys, refs):
        assert np.array_equal(bits(Y.cpu().numpy()), bits(ref))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        chain()
    for Y in Ys:
        Y.zero_()
    g.replay()
    torch.cuda.synchronize()
    for Y, ref in zip(Ys, refs):
        assert np.array_equal(bits(Y.cpu().numpy()), bits(ref))


@pytest.mark.parametrize("R", [1, 2, 4])
@pytest.mark.parametrize("M,K,N,seed", [(3, 3584, 300, 20), (8, 18944, 129, 21), (16, 1024, 777, 22),
                                        (25, 2304, 260, 23)])
def test_qmma_tiles_per_warp(w4, orc, ops, R, M, K, N, seed):
    """Every tiles-per-warp choice (boxes interleaved over R warp groups)
    gives the oracle's bits; with e4m3 operands 4 tiles a warp exist up to 16
    rows (past that the call takes the next kernel)."""
    w4.w4a8_set_tuning(qmma_tiles_per_warp=R, qmma_max_m=32, qmma_operands=ops)
    if R == 4 and M > 16 and ops == 2:  # no such e4m3 kernel: the call goes to the tensor cores
        assert w4.w4a8_plan_info(M, K, N)["kernel"] == 1
        return
    assert w4.w4a8_plan_info(M, K, N)["threads_per_row"] == R
    check(w4, orc, M, K, N, 990 + seed)
