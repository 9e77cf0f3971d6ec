"""w4a8_linear_noalloc: the fused W4A8 linear for callers that cannot provide
workspace memory (code paths that must not allocate device memory, because an
allocation can synchronise the device and take unbounded time).  Its split-K
scratch is a static per-GPU array inside the library.

Checked through the C ABI against w4a8_linear with an ordinary workspace: the
results must be bit-identical, on two calls in a row (the second call reuses
the scratch the first one left behind).  This file is collected last so that a
run stopping at its first failure has already run every other test; it also
passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import synth  # noqa: E402

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 4 << 20  # W4A8_NOALLOC_SCRATCH in include/w4a8.h


@pytest.fixture(scope="module")
def w4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_weight_quantized_w4a8_gb300 as m
    m.build()
    m.w4a8_set_tuning(reset=True)
    yield m
    m.w4a8_set_tuning(reset=True)


def make_inputs(w4, M, K, N, seed):
    W = torch.from_numpy(synth.normal(seed, (N, K), 0.02)).cuda()
    Wq, sw = w4.w4_quantize_weights(W)
    X = torch.from_numpy(synth.activation(seed + 9, M, K, outlier_frac=0.001)).cuda()
    return X, Wq, sw


def call_noalloc(w4, X, Wq, sw, Y):
    """Straight through the C ABI (ctypes), no Python-side allocation."""
    M, K = X.shape
    N = Wq.shape[0]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return w4.lib().w4a8_linear_noalloc(X.data_ptr(), M, K, Wq.data_ptr(), sw.data_ptr(), N,
                                        Y.data_ptr(), 0, stream)


@pytest.mark.parametrize("M,K,N,splits", [(1, 3584, 3000, 4), (3, 18944, 500, 3), (1, 896, 512, 0),
                                          (8, 1024, 700, 16)])
def test_noalloc_matches_workspace_path_twice(w4, M, K, N, splits):
    # the reference call takes the same dp4a plan the entry point launches,
    # so `need` is that plan's scratch and the comparison is plan for plan
    w4.w4a8_set_tuning(force_splits=splits, mma_min_m=65, rowdot_max_m=1, qmma_max_m=1)
    try:
        need = w4.w4a8_workspace_bytes(M, K, N)
        assert need <= SCRATCH_BYTES
        if splits:
            assert need > 0  # the split-K scratch is really exercised
        ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
        for rep in range(2):
            X, Wq, sw = make_inputs(w4, M, K, N, 300 + rep)
            ref = w4.w4a8_linear(X, Wq, sw, ws=ws)
            Y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
            st = call_noalloc(w4, X, Wq, sw, Y)
            assert st == 0, w4.w4a8_last_error()
            torch.cuda.synchronize()
            assert np.array_equal(Y.cpu().numpy().view(np.uint32), ref.cpu().numpy().view(np.uint32))
    finally:
        w4.w4a8_set_tuning(reset=True)
    assert w4.w4a8_device_error() == 0


def test_noalloc_rejects_plans_beyond_the_static_scratch(w4):
    M, K, N = 8, 4096, 10000
    w4.w4a8_set_tuning(force_splits=16, mma_min_m=65, rowdot_max_m=1, qmma_max_m=1)  # the dp4a plan the entry point uses
    try:
        assert w4.w4a8_workspace_bytes(M, K, N) > SCRATCH_BYTES
        X = torch.zeros((M, K), dtype=torch.float16, device="cuda")
        Wq = torch.zeros((N, K // 2), dtype=torch.uint8, device="cuda")
        sw = torch.zeros((N,), dtype=torch.float32, device="cuda")
        Y = torch.zeros((M, N), dtype=torch.float32, device="cuda")
        assert call_noalloc(w4, X, Wq, sw, Y) == 4  # W4A8_ERR_WORKSPACE
        assert "static scratch" in w4.w4a8_last_error()
    finally:
        w4.w4a8_set_tuning(reset=True)


@pytest.mark.parametrize("M,K,N", [(2, 3584, 18944), (3, 3584, 1000), (4, 3584, 18944),
                                   (8, 18944, 3584), (8, 3584, 152064), (5, 896, 77),
                                   (2, 3584, 152064)])
def test_noalloc_takes_the_routed_kernel(w4, M, K, N):
    """With the default routing, 2..8 rows run the kernel w4a8_linear picks
    (row-per-thread, tensor cores, or on lm_head-sized matrices at 2..4 rows
    the warp-level MMA kernel's persistent plan) inside the static scratch,
    twice in a row, bit-identical to w4a8_linear with its own workspace."""
    w4.w4a8_set_tuning(reset=True)
    need = w4.w4a8_workspace_bytes(M, K, N)
    assert 0 < need <= SCRATCH_BYTES
    assert w4.w4a8_plan_info(M, K, N)["kernel"] in ((3,) if (M <= 4 and N >= 77824) else (1, 2))
    for rep in range(2):
        X, Wq, sw = make_inputs(w4, M, K, N, 320 + rep)
        ref = w4.w4a8_linear(X, Wq, sw)
        Y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        st = call_noalloc(w4, X, Wq, sw, Y)
        assert st == 0, w4.w4a8_last_error()
        torch.cuda.synchronize()
        assert np.array_equal(Y.cpu().numpy().view(np.uint32), ref.cpu().numpy().view(np.uint32))
    assert w4.w4a8_device_error() == 0
