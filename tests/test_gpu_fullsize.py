"""Full-size workloads in the launch configuration the benchmark times, checked
against the CPU oracle on EVERY output element.

Weights are drawn on the host by the C twin of the seeded generator
(synth.normal_host: the same bits as the numpy definition), quantized by the
oracle (row chunks on host threads) and, separately, uploaded and quantized
by the GPU; packed codes and scales are compared in full, then every output
of the GPU linear against the oracle's.

* Qwen2-7B-shaped decode linear set, M=1, W4A8 (q, k, v, o, gate, up, down,
  lm_head), activations with 0.1% x20 outliers, fused activation
  quantization, programmatic dependent launch; and the same step as the
  benchmark launches it (q/k/v and gate/up grouped).
* The full 28-layer decode step's own weights and activations (seeds
  1000 * (layer + 1) + index) for layers 0, 13 and 27, all five launches of
  each layer as the benchmark runs them.
* Skinny-batch sweep on gate and down, M in {1, 2, 4, 8, 16, 32, 64}, and
  lm_head at 2, 3, 4, 8 and 16 rows.
* ChatGLM2-6B-shaped W8A16 GEMVs (every output within the tolerance).
"""
import concurrent.futures as cf
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import synth  # noqa: E402

pytestmark = pytest.mark.gpu

# (name, K, N): in-features K, out-features N
QWEN2_7B_SET = [("q", 3584, 3584), ("k", 3584, 512), ("v", 3584, 512), ("o", 3584, 3584),
                ("gate", 3584, 18944), ("up", 3584, 18944), ("down", 18944, 3584),
                ("lm_head", 3584, 152064)]
LAUNCHES = [("qkv", ("q", "k", "v")), ("o", ("o",)), ("gate_up", ("gate", "up")),
            ("down", ("down",)), ("lm_head", ("lm_head",))]
CHATGLM2_W8A16 = [("h_to_4h", 4096, 27392), ("qkv", 4096, 4608), ("4h_to_h", 13696, 4096)]
WEIGHT_SEED0 = 1000
ACT_SEED_OFFSET = 500
OUTLIER_FRAC = 0.001
NAMES = [s[0] for s in QWEN2_7B_SET]
THREADS = os.cpu_count() or 4


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


def bits(a):
    return np.ascontiguousarray(a).view(np.uint32)


def chunks(n, parts):
    step = max(1, -(-n // parts))
    return [(i, min(n, i + step)) for i in range(0, n, step)]


def oracle_quantize(orc, W):
    """orc.w4_quantize over row chunks on host threads (rows are independent)."""
    N, K = W.shape
    Wq = np.empty((N, K // 2), np.uint8)
    sw = np.empty(N, np.float32)

    def one(c):
        q, s = orc.w4_quantize(W[c[0]:c[1]])
        Wq[c[0]:c[1]], sw[c[0]:c[1]] = q, s

    with cf.ThreadPoolExecutor(THREADS) as ex:
        list(ex.map(one, chunks(N, 4 * THREADS)))
    return Wq, sw


def oracle_linear(orc, X, Wq, sw):
    """orc.w4a8_linear over output-row chunks on host threads: (Y, Xq, sa)."""
    N = Wq.shape[0]
    Y = np.empty((X.shape[0], N), np.float32)
    first = {}

    def one(c):
        y, xq, sa, _ = orc.w4a8_linear(X, Wq[c[0]:c[1]], sw[c[0]:c[1]])
        Y[:, c[0]:c[1]] = y
        if c[0] == 0:
            first["xq"], first["sa"] = xq, sa

    with cf.ThreadPoolExecutor(THREADS) as ex:
        list(ex.map(one, chunks(N, 4 * THREADS)))
    return Y, first["xq"], first["sa"]


_weights = {}


def weights(w4, orc, seed, N, K):
    """(Wq, sw) on the GPU and (Wq_ref, sw_ref) from the oracle for the
    weight tensor normal(seed, (N, K), 0.02); the GPU quantizer is checked
    against the oracle on every byte and scale.  Cached per tensor."""
    key = (seed, N, K)
    if key not in _weights:
        W = synth.normal_host(seed, (N, K), 0.02)
        Wd = torch.from_numpy(W).cuda()
        Wq, sw = w4.w4_quantize_weights(Wd)
        del Wd
        Wq_ref, sw_ref = oracle_quantize(orc, W)
        del W
        assert np.array_equal(Wq.cpu().numpy(), Wq_ref), "packed weights differ (seed %d)" % seed
        assert np.array_equal(bits(sw.cpu().numpy()), bits(sw_ref)), "weight scales differ (seed %d)" % seed
        if len(_weights) > 24:
            _weights.clear()
        _weights[key] = (Wq, sw, Wq_ref, sw_ref)
    return _weights[key]


def run_w4(w4, orc, K, N, M, seed, flags):
    Wq, sw, Wq_ref, sw_ref = weights(w4, orc, seed, N, K)
    X = synth.activation(seed + ACT_SEED_OFFSET, M, K, outlier_frac=OUTLIER_FRAC)
    Xq = torch.empty((M, K), dtype=torch.int8, device="cuda")
    sa = torch.empty((M,), dtype=torch.float32, device="cuda")
    Y = w4.w4a8_linear(torch.from_numpy(X).cuda(), Wq, sw, Xq_out=Xq, sa_out=sa, flags=flags)
    torch.cuda.synchronize()
    Y_ref, Xq_ref, sa_ref = oracle_linear(orc, X, Wq_ref, sw_ref)
    assert np.array_equal(Xq.cpu().numpy(), Xq_ref)
    assert np.array_equal(bits(sa.cpu().numpy()), bits(sa_ref))
    Yh = Y.cpu().numpy()
    bad = np.argwhere(bits(Yh) != bits(Y_ref))
    assert bad.size == 0, ("%d outputs differ" % len(bad), bad[:5])
    assert np.isfinite(Yh).all()


@pytest.mark.parametrize("idx", range(len(QWEN2_7B_SET)), ids=NAMES)
def test_qwen2_7b_linear_set_m1(w4, orc, idx):
    name, K, N = QWEN2_7B_SET[idx]
    run_w4(w4, orc, K, N, 1, WEIGHT_SEED0 + idx, flags=w4.LAUNCH_PDL)
    assert w4.w4a8_device_error() == 0


def run_step(w4, orc, wseed, aseed, launches, check_every=True):
    """The launches of one decode layer (q/k/v and gate/up grouped, PDL) on
    weights wseed(i) and activations aseed(first member); every output is
    compared with the oracle."""
    Wd, refs, Xs, Ys = {}, {}, {}, {}
    for lname, members in launches:
        for n in members:
            i = NAMES.index(n)
            _, K, N = QWEN2_7B_SET[i]
            Wq, sw, Wq_ref, sw_ref = weights(w4, orc, wseed(i), N, K)
            Wd[n] = (Wq, sw)
            refs[n] = (Wq_ref, sw_ref)
        K = QWEN2_7B_SET[NAMES.index(members[0])][1]
        Xs[lname] = synth.activation(aseed(NAMES.index(members[0])), 1, K, outlier_frac=OUTLIER_FRAC)
    for lname, members in launches:
        Xd = torch.from_numpy(Xs[lname]).cuda()
        if len(members) == 1:
            Wq, sw = Wd[members[0]]
            Ys[members[0]] = w4.w4a8_linear(Xd, Wq, sw, flags=w4.LAUNCH_PDL)
        else:
            out = w4.w4a8_linear_grouped(Xd, [Wd[n][0] for n in members], [Wd[n][1] for n in members],
                                         flags=w4.LAUNCH_PDL)
            Ys.update(dict(zip(members, out)))
    torch.cuda.synchronize()
    for lname, members in launches:
        for n in members:
            Y_ref = oracle_linear(orc, Xs[lname], *refs[n])[0]
            assert np.array_equal(bits(Ys[n].cpu().numpy()), bits(Y_ref)), n
    assert w4.w4a8_device_error() == 0


def test_decode_step_as_benchmarked(w4, orc):
    """One step exactly as bench.py runs it (grouped q/k/v and gate/up, PDL),
    every output of every linear checked against the oracle."""
    import bench
    assert [l[0] for l in bench.LINEARS] == NAMES and bench.LAUNCHES == LAUNCHES
    run_step(w4, orc, lambda i: WEIGHT_SEED0 + i, lambda i: WEIGHT_SEED0 + i + ACT_SEED_OFFSET, LAUNCHES)


@pytest.mark.parametrize("layer", [0, 13, 27])
def test_decode_28_layers_own_inputs(w4, orc, layer):
    """Layers of the 28-layer decode step at their own seeds (weights
    1000 * (layer + 1) + index, activations that + 500, as the benchmark
    draws them): q/k/v, o, gate/up and down launched as the benchmark does,
    every output element against the oracle."""
    import bench
    assert bench.DECODE_LAYERS == 28
    base = 1000 * (layer + 1)
    run_step(w4, orc, lambda i: base + i, lambda i: base + i + ACT_SEED_OFFSET, LAUNCHES[:-1])


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16, 32, 64])
@pytest.mark.parametrize("name", ["gate", "down"])
def test_skinny_batch_sweep(w4, orc, M, name):
    idx = NAMES.index(name)
    _, K, N = QWEN2_7B_SET[idx]
    run_w4(w4, orc, K, N, M, WEIGHT_SEED0 + idx, flags=w4.LAUNCH_PDL)


@pytest.mark.parametrize("M", [2, 3, 4, 8, 16])
def test_lm_head_small_batches(w4, orc, M):
    """lm_head at small batch sizes: 2..4 rows on the warp-level MMA kernel
    (persistent CTAs, two per SM, walking the 1188 tiles), more on the e4m3
    tensor cores (a 1188-tile grid in several waves)."""
    idx = NAMES.index("lm_head")
    _, K, N = QWEN2_7B_SET[idx]
    assert w4.w4a8_plan_info(M, K, N)["kernel"] == (3 if M <= 4 else 1)
    run_w4(w4, orc, K, N, M, WEIGHT_SEED0 + idx, flags=w4.LAUNCH_PDL)


def test_batch_above_limit_rejected(w4):
    X = torch.zeros((65, 3584), dtype=torch.float16, device="cuda")
    Wq = torch.zeros((64, 1792), dtype=torch.uint8, device="cuda")
    sw = torch.zeros((64,), dtype=torch.float32, device="cuda")
    with pytest.raises(w4.W4A8Error) as e:
        w4.w4a8_linear(X, Wq, sw)
    assert e.value.status == 3


@pytest.mark.parametrize("idx", range(len(CHATGLM2_W8A16)), ids=[s[0] for s in CHATGLM2_W8A16])
def test_chatglm2_w8a16(w4, orc, idx):
    name, K, N = CHATGLM2_W8A16[idx]
    seed = 2000 + idx
    W = synth.normal_host(seed, (N, K), 0.02)
    Wq8, sw16 = w4.w8_quantize_weights(torch.from_numpy(W).cuda())
    X = synth.activation(seed + ACT_SEED_OFFSET, 1, K)
    Y = w4.w8a16_gemv(torch.from_numpy(X).cuda(), Wq8, sw16, flags=w4.LAUNCH_PDL)
    torch.cuda.synchronize()
    Wq_ref = np.empty((N, K), np.int8)
    sw_ref = np.empty(N, np.uint16)
    Y_ref = np.empty((1, N), np.float64)

    def one(c):
        q, s = orc.w8_quantize(W[c[0]:c[1]])
        Wq_ref[c[0]:c[1]], sw_ref[c[0]:c[1]] = q, s.view(np.uint16)
        Y_ref[:, c[0]:c[1]] = orc.w8a16_ref(X, q, s)

    with cf.ThreadPoolExecutor(THREADS) as ex:
        list(ex.map(one, chunks(N, 4 * THREADS)))
    assert np.array_equal(Wq8.cpu().numpy(), Wq_ref)
    assert np.array_equal(sw16.cpu().numpy().view(np.uint16), sw_ref)
    got = Y.cpu().numpy().astype(np.float64)
    err = np.abs(got - Y_ref)
    assert np.sqrt((err ** 2).sum() / (Y_ref ** 2).sum()) <= 5e-4
    assert np.all(err <= 1e-3 * (np.abs(Y_ref) + 1))
