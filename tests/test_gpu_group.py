"""Group-wise INT4 scales: CUDA path vs the CPU oracle through the C ABI.

Codes, scales and the quantized activation are bit-exact, and so is Y: the
library fixes the order of the group-scale arithmetic by K and the group
size alone (exact int32 group sums folded in ascending order with one fused
multiply-add each inside chunks of max(gs, 1024) codes, chunk results added
in ascending order, then times s_a), and the oracle evaluates that order
(oracle_w4a8g_f32).  Y is also within the recursive-summation bound of the
oracle's binary64 value, and a row gives the same bits at every batch size,
split count and kernel.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import guards  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402

pytestmark = pytest.mark.gpu

U = 2.0 ** -24

# tuning of each routing: the default (one-thread-per-row kernel for 1..8
# rows, tensor cores above), one launch per 8 rows on the one-thread-per-row
# kernel, and the tensor cores from 3 rows
PATHS = {"default": {}, "row_groups": dict(rowdot_max_m=1, mma_min_m=65),
         "tensor_cores": dict(rowdot_max_m=1)}


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


def assert_exact(Y, Y_ref):
    Y, Y_ref = np.ascontiguousarray(Y, np.float32), np.ascontiguousarray(Y_ref, np.float32)
    bad = np.argwhere(bits(Y) != bits(Y_ref))
    assert bad.size == 0, (len(bad), bad[:5], Y[tuple(bad[0])], Y_ref[tuple(bad[0])])


def assert_within_bound(Y, Y64, B, K, gs):
    """The fixed order's rounding bound: (groups per chunk + chunks + 1)
    roundings of at most 2^-24 relative each, in the magnitude B."""
    L = max(gs, 1024)
    n_round = L // gs + (K + L - 1) // L + 1
    err = np.abs(Y.astype(np.float64) - Y64)
    assert np.all(err <= n_round * U * 1.001 * B + 1e-300)


def route(w4, path, M, gs):
    """Sets the tuning of a routing; False when it cannot serve the call."""
    if path == "tensor_cores" and (M < 3 or gs % 128 or gs > 16384):
        return False
    w4.w4a8_set_tuning(**PATHS[path])
    return True


def make_operands(M, K, N, gs, seed):
    W = synth.normal(seed, (N, K), 0.02)
    W[1 % N] = 0.0                        # a zero row: every scale 0, outputs 0
    if K // gs > 1:
        W[0, gs:2 * gs] = 0.0             # a zero group inside a non-zero row
    X = synth.activation(seed + 7, M, K, outlier_frac=0.001)
    if M > 1:
        X[M - 1] = 0                      # a zero activation row: s_a 0, outputs 0
    return W, X


def check_group(w4, orc, M, K, N, gs, seed, fused=True, flags=0):
    W, X = make_operands(M, K, N, gs, seed)
    Wq_ref, sg_ref = orc.w4g_quantize(W, gs)
    Y_ref, Xq_ref, sa_ref = orc.w4a8g_linear_f32(X, Wq_ref, sg_ref, gs)

    Wq, sg = w4.w4g_quantize_weights(to_dev(W), gs)
    assert np.array_equal(Wq.cpu().numpy(), Wq_ref)
    assert np.array_equal(bits(sg.cpu().numpy()), bits(sg_ref))
    gY = guards.out((M, N), torch.float32)
    gXq, gsa = guards.out((M, K), torch.int8), guards.out((M,), torch.float32)
    gws = guards.workspace(w4.w4a8g_workspace_bytes(M, K, N, gs))
    Xq, sa = gXq.t, gsa.t
    if fused:
        Y = w4.w4a8g_linear(to_dev(X), Wq, sg, gs, Y=gY.t, Xq_out=Xq, sa_out=sa,
                            ws=guards.t(gws), flags=flags)
    else:
        w4.act_quantize_i8(to_dev(X), Xq=Xq, sa=sa)
        Y = w4.w4a8g_gemv(Xq, sa, Wq, sg, gs, Y=gY.t, ws=guards.t(gws), flags=flags)
    guards.check_all(gY, gXq, gsa, gws)
    assert np.array_equal(Xq.cpu().numpy(), Xq_ref)
    assert np.array_equal(bits(sa.cpu().numpy()), bits(sa_ref))
    Yh = Y.cpu().numpy()
    assert_exact(Yh, Y_ref)
    Y64, B = orc.w4a8g_ref(Xq_ref, sa_ref, Wq_ref, sg_ref, gs)
    assert_within_bound(Yh, Y64, B, K, gs)
    assert not Yh[:, 1 % N].any()
    if M > 1:
        assert not Yh[M - 1].any()
    return Yh


@pytest.mark.parametrize("N,K,gs,seed", [(512, 896, 128, 0), (37, 3584, 128, 1), (5, 32, 32, 2),
                                         (64, 18944, 128, 3), (9, 4096, 4096, 4), (17, 1024, 64, 5),
                                         (3, 2048, 256, 6)])
def test_w4g_quantize(w4, orc, N, K, gs, seed):
    W = synth.normal(seed, (N, K), 0.02)
    W[0, :gs] = 0.0
    W[N - 1, K - 1] *= 30.0
    Wq_ref, sg_ref = orc.w4g_quantize(W, gs)
    Wq, sg = w4.w4g_quantize_weights(to_dev(W), gs)
    torch.cuda.synchronize()
    assert np.array_equal(Wq.cpu().numpy(), Wq_ref)
    assert np.array_equal(bits(sg.cpu().numpy()), bits(sg_ref))


def test_w4g_quantize_equals_rowwise_at_group_k(w4):
    W = to_dev(synth.normal(8, (33, 4096), 0.02))
    Wq_r, sw = w4.w4_quantize_weights(W)
    Wq_g, sg = w4.w4g_quantize_weights(W, 4096)
    torch.cuda.synchronize()
    assert torch.equal(Wq_r, Wq_g)
    assert torch.equal(sg[:, 0], sw) and not sg[:, 1:].any()


GROUP_SHAPES = [
    # M, K, N, gs, seed: several tiles, ragged N, every group size, odd group counts
    (1, 896, 512, 128, 10), (1, 3584, 300, 128, 11), (1, 18944, 129, 128, 12),
    (2, 3584, 260, 64, 13), (3, 1024, 77, 32, 14), (4, 3584, 1000, 256, 15),
    (5, 896, 33, 128, 16), (8, 2048, 200, 512, 17), (1, 32, 7, 32, 18), (1, 4096, 64, 4096, 19),
    (11, 896, 100, 128, 20), (64, 384, 96, 128, 21),
    (2, 3584, 1000, 128, 800),   # two chunks of 1024 and a partial one
    (6, 4096, 40000, 512, 804),  # many tiles, one piece each
    (7, 288, 7, 32, 805),        # a partial last box
    (8, 18944, 700, 128, 806),   # long rows, chunk-aligned pieces
    (8, 4096, 64, 4096, 807),    # one group per row: one chunk
    (4, 2048, 5, 1024, 808),     # groups of a whole chunk
    (3, 8192, 40, 2048, 809),    # chunks of one group larger than 1024 codes
    (20, 3072, 300, 32, 810),    # batches of 8, 8, 4 rows (groups the tensor cores do not take)
]


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("M,K,N,gs,seed", GROUP_SHAPES)
def test_w4a8g_linear(w4, orc, M, K, N, gs, seed, path):
    if not route(w4, path, M, gs):
        pytest.skip("the routing does not serve this call")
    check_group(w4, orc, M, K, N, gs, seed, fused=True)


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("M,K,N,gs,seed", GROUP_SHAPES[:6] + GROUP_SHAPES[10:14])
def test_w4a8g_gemv_unfused(w4, orc, M, K, N, gs, seed, path):
    if not route(w4, path, M, gs):
        pytest.skip("the routing does not serve this call")
    check_group(w4, orc, M, K, N, gs, seed, fused=False)


# the tensor-core path: groups of whole 128-code stages, 3..64 rows; small N
# splits K into pieces of whole chunks (chunk sums added by the last CTA)
MMA_GROUP_SHAPES = [
    (3, 3584, 300, 128, 90), (16, 3584, 1000, 128, 91), (64, 896, 129, 128, 92),
    (33, 2048, 257, 256, 93), (8, 18944, 200, 128, 94), (5, 4096, 64, 4096, 95),
    (24, 1024, 4096, 512, 96), (40, 3072, 130, 1024, 97), (17, 4096, 300, 2048, 98),
]


@pytest.mark.parametrize("M,K,N,gs,seed", MMA_GROUP_SHAPES)
@pytest.mark.parametrize("fused", [True, False])
def test_w4a8g_tensor_cores(w4, orc, M, K, N, gs, seed, fused):
    w4.w4a8_set_tuning(**PATHS["tensor_cores"])
    p = w4.w4a8g_plan_info(M, K, N, gs)
    assert p["kernel"] == 1
    check_group(w4, orc, M, K, N, gs, seed, fused=fused)


def test_w4a8g_tensor_cores_split_and_whole(w4, orc):
    """The plans of the tensor-core group path include split K (few tiles)
    and whole K (many tiles, or one chunk)."""
    w4.w4a8_set_tuning(**PATHS["tensor_cores"])
    assert w4.w4a8g_plan_info(8, 18944, 200, 128)["splits"] > 1
    assert w4.w4a8g_plan_info(24, 1024, 4096, 512)["splits"] == 1
    assert w4.w4a8g_plan_info(64, 3584, 40000, 128)["splits"] == 1


@pytest.mark.parametrize("splits", [1, 2, 3, 5, 16])
@pytest.mark.parametrize("fused", [True, False])
def test_w4a8g_split_k(w4, orc, splits, fused):
    """K pieces of whole chunks, every count up to one chunk per piece: the
    same bits as the oracle (the chunk sums are added in chunk order by the
    CTA that finishes a tile last)."""
    w4.w4a8_set_tuning(force_splits=splits)
    for (M, K, N, gs, seed) in [(2, 3584, 300, 128, 30), (1, 18944, 70, 64, 40), (5, 8192, 200, 2048, 50)]:
        p = w4.w4a8g_plan_info(M, K, N, gs)
        nch = -(-K // max(gs, 1024))
        assert p["kernel"] == 2 and p["splits"] == -(-nch // -(-nch // min(splits, nch)))
        check_group(w4, orc, M, K, N, gs, seed + splits, fused=fused)


def test_w4a8g_same_bits_at_every_batch(w4, orc):
    """One activation row inside batches of 1 to 64 rows, on every kernel
    and split count: the same output bits, those of the oracle."""
    K, N, gs = 3584, 1000, 128
    W = synth.normal(120, (N, K), 0.02)
    Xb = synth.activation(121, 64, K, outlier_frac=0.001)
    Wq_ref, sg_ref = orc.w4g_quantize(W, gs)
    Y_ref = orc.w4a8g_linear_f32(Xb[:1], Wq_ref, sg_ref, gs)[0]
    Wq, sg = w4.w4g_quantize_weights(to_dev(W), gs)
    seen = set()
    for M in (1, 2, 5, 8, 9, 16, 40, 64):
        for path in PATHS:
            for splits in (0, 1, 4):
                if not route(w4, path, M, gs):
                    continue
                w4.w4a8_set_tuning(force_splits=splits, **PATHS[path])
                p = w4.w4a8g_plan_info(M, K, N, gs)
                seen.add((p["kernel"], p["splits"]))
                Y = w4.w4a8g_linear(to_dev(Xb[:M]), Wq, sg, gs)
                assert_exact(Y.cpu().numpy()[:1], Y_ref)
    assert {k for k, _ in seen} == {1, 2} and {P for _, P in seen} >= {1, 4}


def test_w4a8g_exact_powers_of_two(w4, orc):
    """Group scales 2^-e (e in 0..3) and integer activations with max 127
    (s_a = 1): every group sum, product and partial sum is exact in fp32,
    so Y equals the oracle's binary64 value bit for bit on every path."""
    M, K, N, gs = 3, 1024, 300, 128
    rng = np.random.Generator(np.random.PCG64(77))
    G = K // gs
    q = rng.integers(-7, 8, size=(N, G, gs))
    q[:, :, 0] = 7 * rng.choice([-1, 1], size=(N, G))
    e = rng.integers(0, 4, size=(N, G, 1))
    W = (q * 2.0 ** -e).reshape(N, K).astype(np.float32)
    X = rng.integers(-126, 127, size=(M, K)).astype(np.float16)
    X[:, 5] = 127
    Wq_ref, sg_ref = orc.w4g_quantize(W, gs)
    Y_ref, B, _, sa_ref = orc.w4a8g_linear(X, Wq_ref, sg_ref, gs)
    assert np.all(sa_ref == 1.0)
    Wq, sg = w4.w4g_quantize_weights(to_dev(W), gs)
    for path in PATHS:
        route(w4, path, M, gs)
        Y = w4.w4a8g_linear(to_dev(X), Wq, sg, gs)
        torch.cuda.synchronize()
        assert np.array_equal(Y.cpu().numpy().astype(np.float64), Y_ref)


def test_w4a8g_deterministic(w4, orc):
    W, X = make_operands(2, 3584, 5000, 128, 60)
    Wq, sg = w4.w4g_quantize_weights(to_dev(W), 128)
    Xd = to_dev(X)
    Y1 = w4.w4a8g_linear(Xd, Wq, sg, 128).clone()
    Y2 = w4.w4a8g_linear(Xd, Wq, sg, 128, flags=w4.LAUNCH_PDL)
    torch.cuda.synchronize()
    assert torch.equal(Y1, Y2)


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("M,K,Ns,gs,splits", [
    (1, 3584, [3584, 512, 512], 128, 0), (1, 3584, [300, 17], 128, 3),
    (2, 896, [64, 100, 33, 5], 128, 0), (4, 1024, [100, 60], 32, 2),
    (8, 3584, [3584, 512, 512], 128, 0), (16, 3584, [1000, 300], 128, 0),
])
def test_w4a8g_linear_grouped(w4, orc, M, K, Ns, gs, splits, path):
    if not route(w4, path, M, gs):
        pytest.skip("the routing does not serve this call")
    w4.w4a8_set_tuning(force_splits=splits, **PATHS[path])
    X = synth.activation(70 + len(Ns), M, K, outlier_frac=0.001)
    Wqs, sgs, refs = [], [], []
    for g, N in enumerate(Ns):
        W = synth.normal(80 + g, (N, K), 0.02)
        Wq_ref, sg_ref = orc.w4g_quantize(W, gs)
        refs.append(orc.w4a8g_linear_f32(X, Wq_ref, sg_ref, gs)[0])
        Wq, sg = w4.w4g_quantize_weights(to_dev(W), gs)
        Wqs.append(Wq)
        sgs.append(sg)
    gws = guards.workspace(w4.w4a8g_workspace_bytes(M, K, sum(Ns), gs))
    Ys = w4.w4a8g_linear_grouped(to_dev(X), Wqs, sgs, gs, ws=guards.t(gws), flags=w4.LAUNCH_PDL)
    torch.cuda.synchronize()
    guards.check_all(gws)
    for Y, Y_ref in zip(Ys, refs):
        assert_exact(Y.cpu().numpy(), Y_ref)


def test_w4a8g_rejects(w4):
    X = torch.zeros((1, 3584), dtype=torch.float16, device="cuda")
    Wq = torch.zeros((8, 1792), dtype=torch.uint8, device="cuda")
    sg = torch.zeros((8, 28), dtype=torch.float32, device="cuda")
    with pytest.raises(w4.W4A8Error):
        w4.w4a8g_linear(X, Wq, torch.zeros((8, 4), dtype=torch.float32, device="cuda"), 3584)  # not a power of two
    with pytest.raises(w4.W4A8Error):
        w4.w4a8g_linear(X, Wq, torch.zeros((8, 4), dtype=torch.float32, device="cuda"), 1024)  # 1024 does not divide 3584
    with pytest.raises(w4.W4A8Error):
        w4.w4a8g_linear(X, Wq, torch.zeros((8, 224), dtype=torch.float32, device="cuda"), 16)  # below 32
    base = torch.zeros(8 * 28 + 4, dtype=torch.float32, device="cuda")
    Y = torch.empty((1, 8), dtype=torch.float32, device="cuda")
    st = w4.lib().w4a8g_linear(X.data_ptr(), 1, 3584, 128, Wq.data_ptr(), base.data_ptr() + 4, 8,
                               Y.data_ptr(), None, None, None, 0, 0, None)
    assert st == w4._binding.ERR_ALIGN  # scale rows must start on 16-byte boundaries


# --------------------------------------------------------------------------
# full size: the Qwen2-7B-shaped linear set at M = 1 with group size 128,
# in the launch configuration of the benchmark (grouped q/k/v and gate/up,
# programmatic dependent launch), checked on sampled rows
# --------------------------------------------------------------------------

QWEN2_LAUNCHES = [[("q", 3584, 3584), ("k", 3584, 512), ("v", 3584, 512)], [("o", 3584, 3584)],
                  [("gate", 3584, 18944), ("up", 3584, 18944)], [("down", 18944, 3584)],
                  [("lm_head", 3584, 152064)]]


def sample_rows(N, seed, n=64):
    rng = np.random.Generator(np.random.PCG64(seed))
    rows = set(rng.choice(N, size=min(n, N), replace=False).tolist()) | {0, N - 1}
    return np.array(sorted(rows), np.int64)


@pytest.mark.parametrize("li", range(len(QWEN2_LAUNCHES)), ids=["qkv", "o", "gate_up", "down", "lm_head"])
def test_w4a8g_qwen2_fullsize(w4, orc, li):
    gs = 128
    mats = QWEN2_LAUNCHES[li]
    K = mats[0][1]
    seed0 = 2000 + 10 * li
    X = synth.activation(seed0 + 500, 1, K, outlier_frac=0.001)
    Wqs, sgs = [], []
    for g, (_, _, N) in enumerate(mats):
        W = synth.normal_gpu(seed0 + g, (N, K), 0.02)
        Wq, sg = w4.w4g_quantize_weights(W, gs)
        del W
        Wqs.append(Wq)
        sgs.append(sg)
    if len(mats) == 1:
        Ys = [w4.w4a8g_linear(to_dev(X), Wqs[0], sgs[0], gs, flags=w4.LAUNCH_PDL)]
    else:
        Ys = w4.w4a8g_linear_grouped(to_dev(X), Wqs, sgs, gs, flags=w4.LAUNCH_PDL)
    torch.cuda.synchronize()
    for g, (_, _, N) in enumerate(mats):
        rows = sample_rows(N, seed0 + g)
        W_rows = synth.weight_rows(seed0 + g, N, K, rows)
        Wq_ref, sg_ref = orc.w4g_quantize(W_rows, gs)
        idx = torch.from_numpy(rows).cuda()
        assert np.array_equal(Wqs[g][idx].cpu().numpy(), Wq_ref)
        assert np.array_equal(bits(sgs[g][idx].cpu().numpy()), bits(sg_ref))
        Y_ref = orc.w4a8g_linear_f32(X, Wq_ref, sg_ref, gs)[0]
        assert_exact(Ys[g].cpu().numpy()[:, rows], Y_ref)


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("M,K,N,gs,seed", [
    (1, 131072, 5, 128, 110),     # longest rows
    (2, 131072, 3, 32, 111),      # longest rows, smallest groups
    (5, 131072, 7, 1024, 112),    # longest rows, one-group chunks
    (4, 131072, 1, 16384, 113),   # largest tensor-core group, one output row
    (8, 131072, 2, 65536, 115),   # two groups per row, each a chunk of its own
    (1, 3584, 1, 128, 114),       # one output row
])
def test_w4a8g_maximum_sizes(w4, orc, M, K, N, gs, seed, path):
    if not route(w4, path, M, gs):
        pytest.skip("the routing does not serve this call")
    check_group(w4, orc, M, K, N, gs, seed)
