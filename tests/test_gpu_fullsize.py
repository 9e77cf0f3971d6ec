"""Full-size workloads in the launch configuration the benchmark times, checked
against the CPU oracle on sampled output rows (the oracle regenerates just
those weight rows from the counter-based generator).

* Qwen2-7B-shaped decode linear set, M=1, W4A8 (q, k, v, o, gate, up, down,
  lm_head), activations with 0.1% x20 outliers, fused activation quantization,
  programmatic dependent launch.
* Skinny-batch sweep on gate and down, M in {1, 2, 4, 8, 16, 32, 64}, and
  lm_head at 3, 8 and 16 rows.
* ChatGLM2-6B-shaped W8A16 GEMVs.
"""
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
CHATGLM2_W8A16 = [("h_to_4h", 4096, 27392), ("qkv", 4096, 4608), ("4h_to_h", 13696, 4096)]
WEIGHT_SEED0 = 1000
ACT_SEED_OFFSET = 500
OUTLIER_FRAC = 0.001


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


def sample_rows(N, seed, n=48):
    rng = np.random.Generator(np.random.PCG64(seed))
    rows = set(rng.choice(N, size=min(n, N), replace=False).tolist()) | {0, N - 1}
    return np.array(sorted(rows), np.int64)


def run_w4(w4, orc, K, N, M, seed, flags):
    W = synth.normal_gpu(seed, (N, K), 0.02)
    Wq, sw = w4.w4_quantize_weights(W)
    rows = sample_rows(N, seed)
    W_rows_dev = W[torch.from_numpy(rows).cuda()].cpu().numpy()
    del W
    X = synth.activation(seed + ACT_SEED_OFFSET, M, K, outlier_frac=OUTLIER_FRAC)
    Xq = torch.empty((M, K), dtype=torch.int8, device="cuda")
    sa = torch.empty((M,), dtype=torch.float32, device="cuda")
    Y = w4.w4a8_linear(torch.from_numpy(X).cuda(), Wq, sw, Xq_out=Xq, sa_out=sa, flags=flags)
    torch.cuda.synchronize()

    W_rows = synth.weight_rows(seed, N, K, rows)
    assert np.array_equal(bits(W_rows_dev), bits(W_rows))  # generator twins agree
    Wq_ref, sw_ref = orc.w4_quantize(W_rows)
    assert np.array_equal(Wq[torch.from_numpy(rows).cuda()].cpu().numpy(), Wq_ref)
    assert np.array_equal(bits(sw.cpu().numpy()[rows]), bits(sw_ref))
    Y_ref, Xq_ref, sa_ref, _ = orc.w4a8_linear(X, Wq_ref, sw_ref)
    assert np.array_equal(Xq.cpu().numpy(), Xq_ref)
    assert np.array_equal(bits(sa.cpu().numpy()), bits(sa_ref))
    assert np.array_equal(bits(Y.cpu().numpy()[:, rows]), bits(Y_ref))
    assert np.isfinite(Y.cpu().numpy()).all()


@pytest.mark.parametrize("idx", range(len(QWEN2_7B_SET)), ids=[s[0] for s in QWEN2_7B_SET])
def test_qwen2_7b_linear_set_m1(w4, orc, idx):
    name, K, N = QWEN2_7B_SET[idx]
    run_w4(w4, orc, K, N, 1, WEIGHT_SEED0 + idx, flags=w4.LAUNCH_PDL)
    assert w4.w4a8_device_error() == 0


def test_decode_step_as_benchmarked(w4, orc):
    """One step exactly as bench.py runs it (grouped q/k/v and gate/up, PDL),
    sampled rows of every output checked against the oracle."""
    import bench
    names = [l[0] for l in bench.LINEARS]
    Wqs, sws, Ys = {}, {}, {}
    for i, (name, K, N) in enumerate(bench.LINEARS):
        W = synth.normal_gpu(bench.WEIGHT_SEED0 + i, (N, K), 0.02)
        Wqs[name], sws[name] = w4.w4_quantize_weights(W)
        del W
    Xs = {}
    for lname, members in bench.LAUNCHES:
        K = bench.LINEARS[names.index(members[0])][1]
        X = synth.activation(bench.activation_seed(members[0]), 1, K, outlier_frac=bench.OUTLIER_FRAC)
        Xs[lname] = X
        Xd = torch.from_numpy(X).cuda()
        if len(members) == 1:
            Ys[members[0]] = w4.w4a8_linear(Xd, Wqs[members[0]], sws[members[0]], flags=w4.LAUNCH_PDL)
        else:
            out = w4.w4a8_linear_grouped(Xd, [Wqs[n] for n in members], [sws[n] for n in members],
                                         flags=w4.LAUNCH_PDL)
            Ys.update(dict(zip(members, out)))
    torch.cuda.synchronize()
    for lname, members in bench.LAUNCHES:
        for name in members:
            i = names.index(name)
            _, K, N = bench.LINEARS[i]
            rows = sample_rows(N, 7000 + i, n=24)
            Wq_ref, sw_ref = orc.w4_quantize(synth.weight_rows(bench.WEIGHT_SEED0 + i, N, K, rows))
            Y_ref = orc.w4a8_linear(Xs[lname], Wq_ref, sw_ref)[0]
            assert np.array_equal(bits(Ys[name].cpu().numpy()[:, rows]), bits(Y_ref)), name
    assert w4.w4a8_device_error() == 0


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16, 32, 64])
@pytest.mark.parametrize("name", ["gate", "down"])
def test_skinny_batch_sweep(w4, orc, M, name):
    idx = [s[0] for s in QWEN2_7B_SET].index(name)
    _, K, N = QWEN2_7B_SET[idx]
    run_w4(w4, orc, K, N, M, WEIGHT_SEED0 + idx, flags=w4.LAUNCH_PDL)


@pytest.mark.parametrize("M", [3, 8, 16])
def test_lm_head_small_batches(w4, orc, M):
    """lm_head at batch sizes that take the row-per-thread kernel (3, 8: a
    1188-tile grid in several waves) and the tensor cores (16)."""
    idx = [s[0] for s in QWEN2_7B_SET].index("lm_head")
    _, K, N = QWEN2_7B_SET[idx]
    assert w4.w4a8_plan_info(M, K, N)["kernel"] == (2 if M <= 8 else 1)
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
    W = synth.normal_gpu(seed, (N, K), 0.02)
    Wq8, sw16 = w4.w8_quantize_weights(W)
    del W
    X = synth.activation(seed + ACT_SEED_OFFSET, 1, K)
    Y = w4.w8a16_gemv(torch.from_numpy(X).cuda(), Wq8, sw16, flags=w4.LAUNCH_PDL)
    torch.cuda.synchronize()
    rows = sample_rows(N, seed)
    Wq_ref, sw_ref = orc.w8_quantize(synth.weight_rows(seed, N, K, rows))
    rdev = torch.from_numpy(rows).cuda()
    assert np.array_equal(Wq8[rdev].cpu().numpy(), Wq_ref)
    assert np.array_equal(sw16[rdev].cpu().numpy().view(np.uint16), sw_ref.view(np.uint16))
    Y_ref = orc.w8a16_ref(X, Wq_ref, sw_ref)
    got = Y.cpu().numpy()[:, rows].astype(np.float64)
    err = np.abs(got - Y_ref)
    assert np.sqrt((err ** 2).sum() / (Y_ref ** 2).sum()) <= 5e-4
    assert np.all(err <= 1e-3 * (np.abs(Y_ref) + 1))
