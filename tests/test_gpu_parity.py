"""CUDA path vs the CPU oracle, element by element, through the C ABI.

W4A8 (quantizers, codes, scales, int32 accumulators, fp32 outputs) must be
bit-exact; W8A16 outputs within the stated tolerance of the fp64 oracle:
relative L2 error <= 5e-4 and |err| <= 1e-3 * (|y| + 1) per element.
Sizes span several tiles and ragged tails; plans are forced through every
split count, threads-per-row setting and a two-stage ring.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import guards  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402

pytestmark = pytest.mark.gpu

W8_REL_L2 = 5e-4
W8_ELEM = 1e-3


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
    w4.w4a8_set_tuning(reset=True)
    yield
    w4.w4a8_set_tuning(reset=True)
    assert w4.w4a8_device_error() == 0


def bits(a):
    a = np.ascontiguousarray(a)
    return a.view(np.uint32 if a.dtype.itemsize == 4 else np.uint16)


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def weights(N, K, seed, sigma=0.02):
    return synth.normal(seed, (N, K), sigma)


def check_w4a8(w4, orc, M, K, N, seed, fused=True, outliers=0.001, flags=0, zero_rows=()):
    W = weights(N, K, seed)
    for r in zero_rows:
        W[r % N] = 0
    X = synth.activation(seed + 7, M, K, outlier_frac=outliers)
    if M > 1:
        X[M - 1] = 0  # a zero activation row: scale 0, codes 0, outputs 0
    Wq_ref, sw_ref = orc.w4_quantize(W)
    Y_ref, Xq_ref, sa_ref, acc_ref = orc.w4a8_linear(X, Wq_ref, sw_ref)

    Wq, sw = w4.w4_quantize_weights(to_dev(W))
    assert np.array_equal(Wq.cpu().numpy(), Wq_ref)
    assert np.array_equal(bits(sw.cpu().numpy()), bits(sw_ref))
    # every output and the workspace sit between guard bytes
    gacc, gY = guards.out((M, N), torch.int32), guards.out((M, N), torch.float32)
    gws = guards.workspace(w4.w4a8_workspace_bytes(M, K, N))
    if fused:
        gXq, gsa = guards.out((M, K), torch.int8), guards.out((M,), torch.float32)
        Xq, sa = gXq.t, gsa.t
        Y = w4.w4a8_linear(to_dev(X), Wq, sw, Y=gY.t, Xq_out=Xq, sa_out=sa, acc_out=gacc.t,
                           ws=guards.t(gws), flags=flags)
    else:
        gXq, gsa = guards.out((M, K), torch.int8), guards.out((M,), torch.float32)
        Xq, sa = w4.act_quantize_i8(to_dev(X), Xq=gXq.t, sa=gsa.t)
        Y = w4.w4a8_gemv(Xq, sa, Wq, sw, Y=gY.t, acc_out=gacc.t, ws=guards.t(gws), flags=flags)
    guards.check_all(gacc, gY, gws, gXq, gsa)
    acc = gacc.t
    assert np.array_equal(Xq.cpu().numpy(), Xq_ref)
    assert np.array_equal(bits(sa.cpu().numpy()), bits(sa_ref))
    assert np.array_equal(acc.cpu().numpy(), acc_ref)
    assert np.array_equal(bits(Y.cpu().numpy()), bits(Y_ref))


# ---------------------------------------------------------------------------
# quantizers
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("N,K,seed", [(512, 896, 0), (37, 3584, 1), (5, 32, 2), (64, 18944, 3),
                                      (300, 64, 4), (1, 131072, 5)])
def test_w4_quantize(w4, orc, N, K, seed):
    W = weights(N, K, seed)
    W[0, 3] = 0.25   # an outlier row
    if N > 2:
        W[2] = 0     # a zero row
    Wq_ref, sw_ref = orc.w4_quantize(W)
    Wq, sw = w4.w4_quantize_weights(to_dev(W))
    assert np.array_equal(Wq.cpu().numpy(), Wq_ref)
    assert np.array_equal(bits(sw.cpu().numpy()), bits(sw_ref))


def test_w4_quantize_golden_rows(w4, orc):
    """The hand-derived closed forms (tests/golden) through the GPU quantizer."""
    import pins
    for c in pins.read_cases("w4_quant_closed_forms.txt"):
        row = np.zeros((1, 32), np.float32)
        vals = [float(v) for v in c["row"]]
        row[0, :len(vals)] = vals
        Wq, sw = w4.w4_quantize_weights(to_dev(row))
        want = [int(b, 16) for b in c["bytes"]]
        assert list(Wq.cpu().numpy()[0, :len(want)]) == want, c["name"]
        assert sw.item() == float(c["scale"][0])


@pytest.mark.parametrize("M,K,seed", [(1, 896, 10), (3, 3584, 11), (8, 18944, 12), (2, 8, 13),
                                      (5, 131072, 14)])
def test_act_quantize(w4, orc, M, K, seed):
    X = synth.activation(seed, M, K, outlier_frac=0.001)
    if M > 1:
        X[1] = 0
    Xq_ref, sa_ref = orc.act_quantize(X)
    Xq, sa = w4.act_quantize_i8(to_dev(X))
    assert np.array_equal(Xq.cpu().numpy(), Xq_ref)
    assert np.array_equal(bits(sa.cpu().numpy()), bits(sa_ref))


@pytest.mark.parametrize("N,K,seed", [(64, 4096, 20), (7, 13696, 21), (33, 16, 22)])
def test_w8_quantize(w4, orc, N, K, seed):
    W = weights(N, K, seed)
    if N > 3:
        W[3] = 0
        W[1] *= 1e-3    # binary16 subnormal scale: clamping is reachable
        W[2, 5] = 1e-5
    Wq_ref, sw_ref = orc.w8_quantize(W)
    Wq8, sw16 = w4.w8_quantize_weights(to_dev(W))
    assert np.array_equal(Wq8.cpu().numpy(), Wq_ref)
    assert np.array_equal(bits(sw16.cpu().numpy()), bits(sw_ref))


# ---------------------------------------------------------------------------
# W4A8 linear
# ---------------------------------------------------------------------------

W4A8_SHAPES = [
    (1, 896, 512, 0),        # the tiny GEMV
    (1, 3584, 37, 1),        # N smaller than a stage
    (1, 3584, 3584, 2),
    (2, 3584, 1000, 3),
    (3, 18944, 77, 4),       # long rows
    (4, 896, 1000, 5),
    (5, 64, 300, 6),
    (8, 3584, 129, 7),
    (1, 32, 1, 8),           # smallest shape
    (7, 96, 33, 9),
    (1, 131072, 5, 10),      # longest rows
    (8, 131072, 3, 11),
    (6, 18944, 600, 12),
    (9, 896, 100, 13),       # row groups: 8 + 1
    (16, 3584, 77, 14),      # 8 + 8
    (37, 256, 50, 15),       # 8 * 4 + 5
    (64, 1024, 40, 16),      # the largest batch
]


@pytest.mark.parametrize("path", ["default", "dp4a"])
@pytest.mark.parametrize("M,K,N,seed", W4A8_SHAPES)
def test_w4a8_linear_fused(w4, orc, M, K, N, seed, path):
    if path == "dp4a":
        w4.w4a8_set_tuning(mma_min_m=65, rowdot_max_m=1, qmma_max_m=1)  # batches of 3+ rows would take the tensor cores
    check_w4a8(w4, orc, M, K, N, seed, fused=True, zero_rows=(1,))


@pytest.mark.parametrize("path", ["default", "dp4a"])
@pytest.mark.parametrize("M,K,N,seed", W4A8_SHAPES[:8] + W4A8_SHAPES[-3:-1])
def test_w4a8_gemv_unfused(w4, orc, M, K, N, seed, path):
    if path == "dp4a":
        w4.w4a8_set_tuning(mma_min_m=65, rowdot_max_m=1, qmma_max_m=1)
    check_w4a8(w4, orc, M, K, N, seed, fused=False)


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("M,K,N,seed", [(1, 18944, 3584, 33), (1, 3584, 18944, 34), (1, 13696, 700, 35)])
def test_w4a8_one_row_plans_fused_and_unfused(w4, orc, M, K, N, seed, fused):
    """The fused and unfused one-row kernels share each shape's plan (ring
    depth, staging, splits): both must run it to completion, bit-exact and
    with no wait timing out, at the long-row and the wide shapes."""
    check_w4a8(w4, orc, M, K, N, seed, fused=fused)
    assert w4.w4a8_device_error() == 0


@pytest.mark.parametrize("splits", [2, 3, 5, 16])
@pytest.mark.parametrize("fused", [True, False])
def test_w4a8_split_k(w4, orc, splits, fused):
    w4.w4a8_set_tuning(force_splits=splits, mma_min_m=65, rowdot_max_m=1, qmma_max_m=1)  # the dp4a kernel's split plans
    for (M, K, N, seed) in [(1, 3584, 700, 30), (3, 18944, 150, 31), (8, 1024, 64, 32)]:
        if (K // 32) < splits:
            continue
        check_w4a8(w4, orc, M, K, N, seed, fused=fused)
        check_w4a8(w4, orc, M, K, N, seed + 1, fused=fused)  # tickets were reset


def tie_activation(M, K, seed):
    """Activation rows whose scale is exactly 1/128 (max|x| = 127/128) and
    whose values are mostly exact half-integers of that scale, (2k+1)/256,
    so x / s_a lands on a tie; the rest are ordinary values."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ties = (2 * rng.integers(0, 127, size=(M, K)) + 1) / 256.0 * rng.choice([-1.0, 1.0], size=(M, K))
    plain = np.clip(rng.normal(0.0, 0.3, size=(M, K)), -0.98, 0.98)
    X = np.where(rng.random((M, K)) < 0.5, ties, plain).astype(np.float16)
    X[:, rng.integers(0, K)] = np.float16(127.0 / 128.0)
    return X


@pytest.mark.parametrize("M,K,N,splits", [(1, 3584, 300, 0), (1, 3584, 300, 3), (2, 896, 200, 0),
                                          (1, 131072, 4, 0)])
def test_w4a8_fused_ties(w4, orc, M, K, N, splits):
    """Ties (and vectors mixing ties with ordinary values) take the exact
    division path of the fused quantizer; every code must match the oracle,
    halves rounded away from zero."""
    if splits:
        w4.w4a8_set_tuning(force_splits=splits)
    X = tie_activation(M, K, 90 + K + M)
    W = weights(N, K, 91)
    Wq_ref, sw_ref = orc.w4_quantize(W)
    Y_ref, Xq_ref, sa_ref, _ = orc.w4a8_linear(X, Wq_ref, sw_ref)
    assert np.all(sa_ref == np.float32(1.0 / 128.0))
    Wq, sw = w4.w4_quantize_weights(to_dev(W))
    Xq = torch.empty((M, K), dtype=torch.int8, device="cuda")
    sa = torch.empty((M,), dtype=torch.float32, device="cuda")
    Y = w4.w4a8_linear(to_dev(X), Wq, sw, Xq_out=Xq, sa_out=sa)
    Xq2, sa2 = w4.act_quantize_i8(to_dev(X))
    torch.cuda.synchronize()
    assert np.array_equal(Xq.cpu().numpy(), Xq_ref)
    assert np.array_equal(Xq2.cpu().numpy(), Xq_ref)
    assert np.array_equal(bits(sa.cpu().numpy()), bits(sa_ref))
    assert np.array_equal(bits(Y.cpu().numpy()), bits(Y_ref))


# ---------------------------------------------------------------------------
# tensor-core path (batches of 16+ rows by default; forced down to 2 here)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,K,N,seed", [(2, 3584, 300, 100), (5, 896, 129, 101), (15, 128, 256, 102),
                                        (16, 18944, 200, 103), (24, 96, 1, 104), (64, 3584, 129, 105)])
@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("ops", [1, 2], ids=["bf16", "e4m3"])
def test_w4a8_tensor_cores(w4, orc, M, K, N, seed, fused, ops):
    w4.w4a8_set_tuning(mma_min_m=2, rowdot_max_m=1, mma_e4m3=ops, qmma_max_m=1)
    assert w4.w4a8_plan_info(M, K, N)["kernel"] == 1
    check_w4a8(w4, orc, M, K, N, seed, fused=fused, zero_rows=(0,))


@pytest.mark.parametrize("ops", [1, 2], ids=["bf16", "e4m3"])
def test_w4a8_tensor_cores_grouped(w4, orc, ops):
    w4.w4a8_set_tuning(mma_min_m=2, rowdot_max_m=1, mma_e4m3=ops, qmma_max_m=1)
    M, K, Ns = 18, 1024, (300, 7, 129)
    X = synth.activation(110, M, K, outlier_frac=0.001)
    Wqs, sws, refs = [], [], []
    for g, N in enumerate(Ns):
        W = weights(N, K, 111 + g)
        Wq_ref, sw_ref = orc.w4_quantize(W)
        refs.append(orc.w4a8_linear(X, Wq_ref, sw_ref)[0])
        Wq, sw = w4.w4_quantize_weights(to_dev(W))
        Wqs.append(Wq)
        sws.append(sw)
    for rep in range(2):
        Ys = w4.w4a8_linear_grouped(to_dev(X), Wqs, sws, flags=w4.LAUNCH_PDL if rep else 0)
        torch.cuda.synchronize()
        for Y, ref in zip(Ys, refs):
            assert np.array_equal(bits(Y.cpu().numpy()), bits(ref))


@pytest.mark.parametrize("ops", [1, 2], ids=["bf16", "e4m3"])
@pytest.mark.parametrize("K", [16384, 32768])
def test_w4a8_tensor_cores_largest_sums(w4, K, ops):
    """Every weight code -8 (nibble 0x8, legal on input) against activation
    codes +127 and -127: each K piece's partial sum reaches 8 * 127 * 16384 =
    16,646,144, just below 2^24, which the fp32 accumulator must hold
    exactly; the pieces are added as int32."""
    w4.w4a8_set_tuning(mma_min_m=2, rowdot_max_m=1, mma_e4m3=ops, qmma_max_m=1)
    M, N = 16, 130
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


def test_w4a8_tensor_cores_match_dp4a(w4, orc):
    """The same call on both paths gives the same bits."""
    M, K, N = 12, 3584, 1000
    W = weights(N, K, 120)
    X = to_dev(synth.activation(121, M, K, outlier_frac=0.001))
    Wq, sw = w4.w4_quantize_weights(to_dev(W))
    w4.w4a8_set_tuning(mma_min_m=65, rowdot_max_m=1, qmma_max_m=1)
    assert w4.w4a8_plan_info(M, K, N)["kernel"] == 0
    Y0 = w4.w4a8_linear(X, Wq, sw)
    w4.w4a8_set_tuning(mma_min_m=2, rowdot_max_m=1, qmma_max_m=1)
    Y1 = w4.w4a8_linear(X, Wq, sw)
    torch.cuda.synchronize()
    assert np.array_equal(bits(Y0.cpu().numpy()), bits(Y1.cpu().numpy()))


@pytest.mark.parametrize("cl", [1, 2, 8, 32, 64, 128, 256])
def test_w4a8_threads_per_row(w4, orc, cl):
    w4.w4a8_set_tuning(force_threads_per_row=cl, rowdot_max_m=1, qmma_max_m=1, mma_min_m=65)  # the dp4a kernel's plans
    for (M, K, N, seed) in [(1, 3584, 300, 40), (2, 2048, 99, 41), (1, 256, 513, 42)]:
        try:
            plan = w4.w4a8_plan_info(M, K, N)
        except w4.W4A8Error:
            continue  # this thread count cannot cover the row with this M
        assert plan["threads_per_row"] == cl
        check_w4a8(w4, orc, M, K, N, seed)


def test_w4a8_two_stage_ring(w4, orc):
    """A two-stage ring wraps many times; mbarrier phases must stay in step."""
    w4.w4a8_set_tuning(ring_bytes=8192)
    assert w4.w4a8_plan_info(1, 3584, 5000)["stages"] == 2
    check_w4a8(w4, orc, 1, 3584, 5000, 50)
    w4.w4a8_set_tuning(ring_bytes=8192, force_splits=3, rowdot_max_m=1, qmma_max_m=1, mma_min_m=65)
    check_w4a8(w4, orc, 2, 18944, 300, 51)


def test_w4a8_pdl_back_to_back_and_graph(w4, orc):
    """Chains of PDL launches sharing one split-K workspace, eager and in a
    CUDA graph replayed twice, give the oracle's results."""
    w4.w4a8_set_tuning(force_splits=4)
    shapes = [(1, 3584, 512, 60), (1, 18944, 256, 61), (1, 3584, 2048, 62), (1, 896, 100, 63)]
    ins, refs = [], []
    for (M, K, N, seed) in shapes:
        W = weights(N, K, seed)
        X = synth.activation(seed + 7, M, K, outlier_frac=0.001)
        Wq_ref, sw_ref = orc.w4_quantize(W)
        refs.append(orc.w4a8_linear(X, Wq_ref, sw_ref)[0])
        ins.append((to_dev(X), to_dev(Wq_ref), to_dev(sw_ref),
                    torch.empty((M, N), dtype=torch.float32, device="cuda")))
    nbytes = max(w4.w4a8_workspace_bytes(M, K, N) for (M, K, N, _) in shapes)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")

    def run():
        for (X, Wq, sw, Y) in ins:
            w4.w4a8_linear(X, Wq, sw, Y=Y, ws=ws, flags=w4.LAUNCH_PDL)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        run()
        run()
    torch.cuda.synchronize()
    for (_, _, _, Y), ref in zip(ins, refs):
        assert np.array_equal(bits(Y.cpu().numpy()), bits(ref))
        Y.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run()
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        for (_, _, _, Y), ref in zip(ins, refs):
            assert np.array_equal(bits(Y.cpu().numpy()), bits(ref))


def test_workspace_checks(w4):
    w4.w4a8_set_tuning(force_splits=2)
    X = torch.zeros((1, 64), dtype=torch.float16, device="cuda")
    Wq = torch.zeros((4, 32), dtype=torch.uint8, device="cuda")
    sw = torch.zeros((4,), dtype=torch.float32, device="cuda")
    need = w4.w4a8_workspace_bytes(1, 64, 4)
    assert need > 0
    small = torch.zeros(need - 256 if need > 256 else 1, dtype=torch.uint8, device="cuda")
    with pytest.raises(w4.W4A8Error) as e:
        w4.w4a8_linear(X, Wq, sw, ws=small)
    assert e.value.status == 4


# ---------------------------------------------------------------------------
# W8A16
# ---------------------------------------------------------------------------

def check_w8a16(w4, orc, M, K, N, seed):
    W = weights(N, K, seed)
    X = synth.activation(seed + 3, M, K)
    Wq_ref, sw_ref = orc.w8_quantize(W)
    Y_ref = orc.w8a16_ref(X, Wq_ref, sw_ref)
    Wq8, sw16 = w4.w8_quantize_weights(to_dev(W))
    assert np.array_equal(Wq8.cpu().numpy(), Wq_ref)
    gY = guards.out((M, N), torch.float32)
    gws = guards.workspace(w4.w8a16_workspace_bytes(M, K, N))
    w4.w8a16_gemv(to_dev(X), Wq8, sw16, Y=gY.t, ws=guards.t(gws))
    guards.check_all(gY, gws)
    Y = gY.t.cpu().numpy().astype(np.float64)
    err = np.abs(Y - Y_ref)
    assert np.sqrt((err ** 2).sum() / max((Y_ref ** 2).sum(), 1e-300)) <= W8_REL_L2
    assert np.all(err <= W8_ELEM * (np.abs(Y_ref) + 1))
    # and the deterministic fp32 summation bound: K roundings of partial sums
    s = sw_ref.astype(np.float64)[None, :]
    absum = np.abs(X.astype(np.float64)) @ np.abs(Wq_ref.astype(np.float64)).T * s
    assert np.all(err <= (K + 2) * 2.0 ** -24 * absum + 1e-30)


@pytest.mark.parametrize("M,K,N,seed", [(1, 4096, 4608, 70), (2, 64, 100, 71), (4, 13696, 50, 72),
                                        (3, 16, 7, 73), (1, 13696, 400, 74), (1, 65536, 3, 75),
                                        (5, 4096, 64, 76), (16, 512, 90, 77), (64, 128, 20, 78)])
def test_w8a16(w4, orc, M, K, N, seed):
    check_w8a16(w4, orc, M, K, N, seed)


@pytest.mark.parametrize("splits", [2, 5])
def test_w8a16_split_k(w4, orc, splits):
    w4.w4a8_set_tuning(force_splits=splits)
    check_w8a16(w4, orc, 1, 4096, 333, 80)
    check_w8a16(w4, orc, 3, 4096, 64, 81)    # M=3 needs pieces of <= 256 granules
    check_w8a16(w4, orc, 1, 13696, 64, 82)


# ---------------------------------------------------------------------------
# generator twin
# ---------------------------------------------------------------------------

def test_gpu_generator_matches_host(w4):
    g = synth.normal_gpu(1234, (3000, 64), 0.02).cpu().numpy()
    assert np.array_equal(bits(g), bits(synth.normal(1234, (3000, 64), 0.02)))
    g = synth.normal_gpu(99, (1000,), 1.0, offset=(1 << 32) - 1000).cpu().numpy()
    assert np.array_equal(bits(g), bits(synth.normal(99, (1000,), 1.0, offset=(1 << 32) - 1000)))


# ---------------------------------------------------------------------------
# grouped launch: several weight matrices sharing the activation
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,K,Ns,splits", [
    (1, 3584, (3584, 512, 512), 0),      # q/k/v shaped
    (3, 896, (5, 77, 300, 1), 0),        # ragged, a one-row segment
    (2, 1024, (33, 600), 3),             # split-K partials span segments
    (1, 3584, (100, 7, 2000), 4),
    (8, 64, (17, 1, 40, 9), 0),
    (1, 18944, (300, 50), 0),
    (12, 512, (40, 7), 0),               # row groups 8 + 4
    (20, 256, (9, 30, 3), 2),
])
def test_w4a8_linear_grouped(w4, orc, M, K, Ns, splits):
    w4.w4a8_set_tuning(force_splits=splits, mma_min_m=65 if splits else 0,
                      rowdot_max_m=1 if splits else 0, qmma_max_m=1)
    X = synth.activation(500 + K, M, K, outlier_frac=0.001)
    refs, Wqs, sws = [], [], []
    for g, N in enumerate(Ns):
        W = weights(N, K, 600 + 7 * g + N)
        Wq_ref, sw_ref = orc.w4_quantize(W)
        refs.append(orc.w4a8_linear(X, Wq_ref, sw_ref)[0])
        Wq, sw = w4.w4_quantize_weights(to_dev(W))
        Wqs.append(Wq)
        sws.append(sw)
    for rep in range(2):
        Ys = w4.w4a8_linear_grouped(to_dev(X), Wqs, sws, flags=w4.LAUNCH_PDL if rep else 0)
        torch.cuda.synchronize()
        for Y, ref in zip(Ys, refs):
            assert np.array_equal(bits(Y.cpu().numpy()), bits(ref))


def test_w4a8_linear_grouped_rejects_bad_groups(w4):
    X = torch.zeros((1, 64), dtype=torch.float16, device="cuda")
    Wq = torch.zeros((4, 32), dtype=torch.uint8, device="cuda")
    sw = torch.zeros((4,), dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        w4.w4a8_linear_grouped(X, [Wq] * 5, [sw] * 5)
    flat = torch.zeros(4 * 32 + 8, dtype=torch.uint8, device="cuda")
    Wq_mis = flat[8:].view(4, 32)                                  # 8 bytes off 16
    with pytest.raises(w4.W4A8Error) as e:
        w4.w4a8_linear_grouped(X, [Wq, Wq_mis], [sw, sw])
    assert e.value.status == 2


def test_prefetch_hint_changes_no_result(w4):
    """The L2 prefetch entry points (a hint for the next launch's weights)
    give the same bits as the plain calls, single and grouped, at one row
    (the dp4a GEMV, which takes the hint) and at 16 rows (which ignores it);
    the hinted range may be shorter or longer than the next matrix."""
    K = 3584
    Wq1, sw1 = w4.w4_quantize_weights(torch.from_numpy(synth.normal(940, (3000, K), 0.02)).cuda())
    Wq2, sw2 = w4.w4_quantize_weights(torch.from_numpy(synth.normal(941, (700, K), 0.02)).cuda())
    for M in (1, 16):
        X = torch.from_numpy(synth.activation(942 + M, M, K, outlier_frac=0.001)).cuda()
        ref = w4.w4a8_linear(X, Wq1, sw1).clone()
        refg = [y.clone() for y in w4.w4a8_linear_grouped(X, [Wq1, Wq2], [sw1, sw2])]
        for nb in (0, 4096, 1 << 20):
            Y = w4.w4a8_linear(X, Wq1, sw1, prefetch=Wq2, prefetch_bytes=nb, flags=w4.LAUNCH_PDL)
            Yg = w4.w4a8_linear_grouped(X, [Wq1, Wq2], [sw1, sw2], prefetch=Wq1, prefetch_bytes=nb)
            torch.cuda.synchronize()
            assert torch.equal(Y, ref)
            assert all(torch.equal(a, b) for a, b in zip(Yg, refg))
    assert w4.w4a8_device_error() == 0


@pytest.mark.parametrize("M", [2, 9, 17, 32])
def test_tensor_cores_many_tiles(w4, M):
    """More 128-row tiles (313 for 40,000 rows) than two per SM, one K piece:
    several waves of CTAs, ragged last tile; every output bit for bit, twice
    in a row."""
    orc = oracle.load()
    K, N = 1024, 40000
    W = synth.normal(960 + M, (N, K), 0.02)
    X = synth.activation(961 + M, M, K, outlier_frac=0.001)
    Wq_ref, sw_ref = orc.w4_quantize(W)
    Y_ref = orc.w4a8_linear(X, Wq_ref, sw_ref)[0]
    w4.w4a8_set_tuning(rowdot_max_m=1, qmma_max_m=1)
    try:
        p = w4.w4a8_plan_info(M, K, N)
        assert p["kernel"] == 1 and p["splits"] == 1 and p["ctas_per_split"] > 2 * 152 * 0.9
        Wq, sw = w4.w4_quantize_weights(torch.from_numpy(W).cuda())
        for _ in range(2):
            gY = guards.out((M, N), torch.float32)
            Y = w4.w4a8_linear(torch.from_numpy(X).cuda(), Wq, sw, Y=gY.t, flags=w4.LAUNCH_PDL)
            torch.cuda.synchronize()
            guards.check_all(gY)
            assert np.array_equal(Y.cpu().numpy().view(np.uint32), Y_ref.view(np.uint32))
    finally:
        w4.w4a8_set_tuning(reset=True)
    assert w4.w4a8_device_error() == 0
