"""Bounded device waits, run out on purpose without faulting or hanging the GPU.

With w4a8_tuning_t.stall_test_us the warp-level MMA kernel's warps (the
kernel is selected with qmma_max_m) first
wait, with that short limit, for a barrier phase that nothing completes (a
flag that nothing sets).  The wait runs out, the kernel records bit 0 in the
device error word, waits (bounded) for the weight copies it already issued
and returns.  The test checks that the call returns, that w4a8_device_error
reports bit 0, and that after re-zeroing the workspace (as the C header asks
after a non-zero error word) the next call on the same workspace is
bit-exact against the oracle.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import synth  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_weight_quantized_w4a8_gb300 as m
    m.build()
    m.w4a8_set_tuning(reset=True)
    yield m
    m.w4a8_set_tuning(reset=True)


@pytest.mark.parametrize("M,K,N", [(6, 3584, 300),      # three tiles, K split (tickets)
                                   (8, 1024, 2000),     # one piece per tile
                                   (4, 1024, 40000)])   # persistent CTAs, several tiles each
def test_stalled_wait_reports_and_next_call_is_exact(w4, M, K, N):
    orc = oracle.load()
    W = synth.normal(1200 + M, (N, K), 0.02)
    X = synth.activation(1300 + M, M, K, outlier_frac=0.001)
    Wq_ref, sw_ref = orc.w4_quantize(W)
    Y_ref = orc.w4a8_linear(X, Wq_ref, sw_ref)[0]
    Wq, sw = w4.w4_quantize_weights(torch.from_numpy(W).cuda())
    Xd = torch.from_numpy(X).cuda()
    assert w4.w4a8_device_error() == 0
    try:
        w4.w4a8_set_tuning(stall_test_us=20000, qmma_max_m=32)  # 20 ms; the warp-level MMA kernel
        assert w4.w4a8_plan_info(M, K, N)["kernel"] == 3
        ws = torch.zeros(w4.w4a8_workspace_bytes(M, K, N), dtype=torch.uint8, device="cuda")
        w4.w4a8_linear(Xd, Wq, sw, ws=ws)           # returns: the wait runs out
        flags = w4.w4a8_device_error()
        assert flags & 1, flags                     # a wait for stage data ran out
        assert not flags & 4, flags                 # the copies in flight all landed
    finally:
        w4.w4a8_set_tuning(reset=True)
    ws.zero_()                                      # as the header asks after an error
    w4.w4a8_set_tuning(qmma_max_m=32)
    for _ in range(2):
        Y = w4.w4a8_linear(Xd, Wq, sw, ws=ws)
        torch.cuda.synchronize()
        assert np.array_equal(Y.cpu().numpy().view(np.uint32), Y_ref.view(np.uint32))
    w4.w4a8_set_tuning(reset=True)
    assert w4.w4a8_device_error() == 0
