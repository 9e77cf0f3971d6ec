"""Host-side checks of the C ABI (no GPU): exported symbols, argument
validation that returns before any CUDA call, and the launch planner."""
import ctypes
import os
import re

import numpy as np
import pytest

import bit_weight_quantized_w4a8_gb300 as w4

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    w4.build()
    return w4.lib()


def header_functions():
    src = open(os.path.join(ROOT, "include", "w4a8.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", src, flags=re.M)))


def test_header_declares_the_entry_points():
    names = header_functions()
    for want in ["w4_quantize_weights", "w8_quantize_weights", "act_quantize_i8", "w4a8_gemv",
                 "w4a8_linear", "w8a16_gemv", "w4a8_workspace_bytes", "w8a16_workspace_bytes",
                 "w4a8_last_error", "w4a8_device_error", "w4a8_set_tuning", "w4a8_plan_info"]:
        assert want in names


def test_every_declared_symbol_is_exported(L):
    for name in header_functions():
        assert hasattr(L, name), name
    assert set(header_functions()) <= set(w4.EXPORTS) | set(header_functions())


def test_binding_covers_header():
    assert set(header_functions()) == set(w4.EXPORTS)


P16 = 0x10000  # a fake, 16-byte aligned address: never dereferenced (checks fail first)


def test_null_pointers_rejected(L):
    assert L.w4_quantize_weights(None, 4, 32, P16, P16, None) == w4._binding.ERR_NULL
    assert L.act_quantize_i8(P16, 1, 32, None, P16, None) == w4._binding.ERR_NULL
    assert L.w4a8_gemv(None, P16, 1, 32, P16, P16, 4, P16, None, None, 0, 0, None) == w4._binding.ERR_NULL
    assert L.w4a8_linear(P16, 1, 32, P16, None, 4, P16, None, None, None, None, 0, 0, None) == w4._binding.ERR_NULL
    assert L.w8a16_gemv(P16, 1, 32, None, P16, 4, P16, None, 0, 0, None) == w4._binding.ERR_NULL
    assert b"NULL" in L.w4a8_last_error()


def test_bad_shapes_rejected(L):
    E = w4._binding.ERR_SHAPE
    assert L.w4_quantize_weights(P16, 4, 48, P16, P16, None) == E          # K % 32
    assert L.w4_quantize_weights(P16, 0, 32, P16, P16, None) == E          # N < 1
    assert L.w8_quantize_weights(P16, 4, 24, P16, P16, None) == E          # K % 16
    assert L.act_quantize_i8(P16, 0, 32, P16, P16, None) == E              # M < 1
    assert L.act_quantize_i8(P16, 1, 12, P16, P16, None) == E              # K % 8
    assert L.w4a8_gemv(P16, P16, 65, 32, P16, P16, 4, P16, None, None, 0, 0, None) == E  # M > 64
    assert L.w4a8_gemv(P16, P16, 1, 40, P16, P16, 4, P16, None, None, 0, 0, None) == E  # K % 32
    assert L.w4a8_gemv(P16, P16, 1, 262144, P16, P16, 4, P16, None, None, 0, 0, None) == E
    assert L.w4a8_linear(P16, 1, 32, P16, P16, 0, P16, None, None, None, None, 0, 0, None) == E
    assert L.w8a16_gemv(P16, 65, 32, P16, P16, 4, P16, None, 0, 0, None) == E  # M > 64
    assert L.w8a16_gemv(P16, 1, 131072, P16, P16, 4, P16, None, 0, 0, None) == E
    assert L.w4a8_workspace_bytes(65, 32, 4) == 0
    assert L.w4a8_linear_noalloc(P16, 9, 32, P16, P16, 4, P16, 0, None) == E  # one launch: M <= 8


def test_misaligned_pointers_rejected(L):
    E = w4._binding.ERR_ALIGN
    assert L.w4_quantize_weights(P16 + 4, 4, 32, P16, P16, None) == E
    assert L.act_quantize_i8(P16, 1, 32, P16 + 8, P16, None) == E
    assert L.w4a8_gemv(P16 + 8, P16, 1, 32, P16, P16, 4, P16, None, None, 0, 0, None) == E
    assert L.w4a8_gemv(P16, P16, 1, 32, P16 + 1, P16, 4, P16, None, None, 0, 0, None) == E
    assert L.w4a8_linear(P16, 1, 32, P16, P16, 4, P16 + 2, None, None, None, None, 0, 0, None) == E
    assert L.w8a16_gemv(P16, 1, 32, P16 + 4, P16, 4, P16, None, 0, 0, None) == E


def test_prefetch_argument_checks(L):
    """The prefetch hint must start on 16 bytes; checked before any launch."""
    E_A = w4._binding.ERR_ALIGN
    assert L.w4a8_linear_prefetch(P16, 1, 32, P16, P16, 4, P16, None, 0, 0, None, P16 + 8, 1024) == E_A
    arr = (ctypes.c_void_p * 1)(P16)
    ns = (ctypes.c_int64 * 1)(4)
    assert L.w4a8_linear_grouped_prefetch(P16, 1, 32, 1, arr, arr, ns, arr, None, 0, 0, None,
                                          P16 + 4, 64) == E_A


def test_grouped_argument_checks(L):
    import ctypes
    arr = (ctypes.c_void_p * 2)(P16, P16)
    ns = (ctypes.c_int64 * 2)(4, 4)
    null_arr = (ctypes.c_void_p * 2)(P16, None)
    assert L.w4a8_linear_grouped(P16, 1, 32, 0, arr, arr, ns, arr, None, 0, 0, None) == w4._binding.ERR_SHAPE
    assert L.w4a8_linear_grouped(P16, 1, 32, 5, arr, arr, ns, arr, None, 0, 0, None) == w4._binding.ERR_SHAPE
    assert L.w4a8_linear_grouped(P16, 1, 32, 2, arr, null_arr, ns, arr, None, 0, 0, None) == w4._binding.ERR_NULL
    bad_n = (ctypes.c_int64 * 2)(4, 0)
    assert L.w4a8_linear_grouped(P16, 1, 32, 2, arr, arr, bad_n, arr, None, 0, 0, None) == w4._binding.ERR_SHAPE
    mis = (ctypes.c_void_p * 2)(P16, P16 + 8)
    assert L.w4a8_linear_grouped(P16, 1, 32, 2, mis, arr, ns, arr, None, 0, 0, None) == w4._binding.ERR_ALIGN
    assert L.w4a8_linear_grouped(None, 1, 32, 2, arr, arr, ns, arr, None, 0, 0, None) == w4._binding.ERR_NULL


def test_tuning_validation():
    with pytest.raises(w4.W4A8Error):
        w4.w4a8_set_tuning(force_splits=17)
    with pytest.raises(w4.W4A8Error):
        w4.w4a8_set_tuning(force_threads_per_row=24)
    with pytest.raises(w4.W4A8Error):
        w4.w4a8_set_tuning(ring_bytes=10 ** 7)
    w4.w4a8_set_tuning(reset=True)


SHAPES = [(1, 896, 512), (1, 3584, 3584), (1, 3584, 512), (1, 3584, 18944), (1, 18944, 3584),
          (1, 3584, 152064), (2, 3584, 18944), (4, 18944, 3584), (8, 3584, 18944),
          (8, 18944, 3584), (3, 32, 1), (1, 64, 100000), (5, 131072, 3), (1, 4096, 7),
          (16, 3584, 18944), (64, 18944, 3584), (33, 896, 100), (32, 3584, 152064),
          (24, 131072, 7), (17, 896, 100), (2, 32, 1)]


@pytest.mark.parametrize("sms", [152, 148, 20, 1])
@pytest.mark.parametrize("w8", [False, True])
def test_plan_invariants(sms, w8):
    for (M, K, N) in SHAPES:
        if w8 and K > 65536:
            continue
        check_any_plan(M, K, N, sms, w8)


def test_plan_invariants_random():
    """The same invariants on 400 seeded random shapes (batch 1..64, K a
    multiple of 32 up to 131072, N up to 300000, 1..160 SMs), under the
    default routing and with the warp-level kernel at every batch it takes
    (both operand types).  Every kernel kind is reached."""
    rng = np.random.default_rng(20261202)
    seen = set()
    tunings = [dict(), dict(qmma_max_m=32), dict(qmma_max_m=32, qmma_operands=1)]
    try:
        for i in range(400):
            M = int(rng.choice([1, 2, 3, 4, 8, rng.integers(1, 65)]))
            K = 32 * int(rng.choice([rng.integers(1, 129), rng.integers(1, 4097)]))
            N = int(rng.choice([rng.integers(1, 5000), rng.integers(1, 300001)]))
            sms = int(rng.choice([152, 148, int(rng.integers(1, 161))]))
            w8 = bool(rng.integers(0, 4) == 0) and K <= 65536 and K % 16 == 0
            tun = tunings[i % len(tunings)]
            w4.w4a8_set_tuning(**tun)
            seen.add(check_any_plan(M, K, N, sms, w8, h16=tun.get("qmma_operands") == 1))
    finally:
        w4.w4a8_set_tuning(reset=True)
    assert seen == {0, 1, 2, 3}, seen


def check_any_plan(M, K, N, sms, w8, h16=False):
    """Checks the plan w4a8_plan_info reports for one call, whichever kernel
    the routing picks (h16: the warp-level kernel has binary16 operands)."""
    p = w4.w4a8_plan_info(M, K, N, w8a16=w8, num_sms=sms)
    if p["kernel"] == 1:
        check_mma_plan(p, M, K, N, sms)
        return 1
    if p["kernel"] == 2:
        check_rowdot_plan(p, M, K, N, sms)
        return 2
    if p["kernel"] == 3:
        check_qmma_plan(p, M, K, N, sms, h16=h16)
        return 3
    M = min(M, 4 if w8 else 8)  # the plan of the first launch of a row-group sequence
    kgran = 16 if w8 else 32
    Gt = K // kgran
    P = p["splits"]
    Gq = -(-Gt // P)
    assert 1 <= P <= 16 and (P - 1) * Gq < Gt
    Cl, S = p["threads_per_row"], p["cols_per_thread"]
    assert Cl & (Cl - 1) == 0 and Cl * S >= Gq and Cl * (S - 1) < Gq
    mt = 1 if M <= 1 else 2 if M <= 2 else 4 if M <= 4 else 8
    assert S <= 8 // mt
    assert p["rows_per_stage"] * Cl == 256
    assert p["grid"] == p["ctas_per_split"] * P
    assert p["ctas_per_split"] <= N
    assert p["rows_per_cta"] * p["ctas_per_split"] >= N
    assert p["rows_per_cta"] <= 4096 or P > 1
    assert 2 <= p["stages"] <= 16
    assert p["stage_bytes"] % 128 == 0 and p["stage_bytes"] >= p["rows_per_stage"] * Gq * 16
    assert p["smem_bytes"] <= 232448
    if P > 1:
        assert p["ws_bytes"] > 0
    return 0


def check_mma_plan(p, M, K, N, sms):
    assert M >= 2
    tiles = -(-N // 128)
    nkb = -(-K // 64)
    P = p["splits"]
    assert p["cols_per_thread"] == -(-M // 16) * 16 <= 64      # the MMA's N
    assert p["ctas_per_split"] == tiles and p["grid"] == tiles * P
    kbp = -(-nkb // P)
    assert kbp <= 256 and (P - 1) * kbp < nkb                   # pieces <= 16384, none empty
    assert p["smem_bytes"] <= 232448
    # the codes, then one int32 slice [M][128] per tile and K piece of a split plan
    assert p["ws_bytes"] >= 4096 + 256 + M * K * 2 + (tiles * P * M * 512 if P > 1 else 0)


def check_qmma_plan(p, M, K, N, sms, h16=False):
    """The warp-level MMA kernel: n-tiles of 8 batch rows (binary16 operands)
    or 4 (e4m3, high and low halves), 16-row tiles per warp R, pieces of
    whole 256-code boxes, every warp's fp32 sums over at most 16384
    (binary16) or 65536 (e4m3) codes, stages of one weight box plus its
    activation slice."""
    assert 2 <= M <= 32
    tiles = -(-N // 128)
    nbox = -(-K // 256)
    rows = 8 if h16 else 4
    NT = -(-M // rows)
    P, R = p["splits"], p["threads_per_row"]
    assert p["cols_per_thread"] == rows * NT and R in (1, 2, 4) and (R < 4 or NT <= 4)
    assert p["ctas_per_split"] == tiles
    # one K piece, more tiles than SMs, the default tiles per warp:
    # persistent CTAs walk the tiles, two per SM up to 2 n-tiles (each within
    # half the SM's shared memory), else one
    persist = P == 1 and tiles > sms and R == (4 if NT <= 4 else 2)
    two = persist and NT <= 2
    assert p["grid"] == (min(tiles, 2 * sms) if two else sms if persist else tiles * P)
    if two:
        assert p["smem_bytes"] <= 233472 // 2 - 1024
    bpp = -(-nbox // P)
    assert (P - 1) * bpp < nbox                                  # no empty piece
    assert -(-bpp // R) * 256 <= (16384 if h16 else 65536)       # exact fp32 sums per warp
    slice_bytes = (4096 if h16 else 2048) * NT
    assert p["stage_bytes"] == 16384 + slice_bytes
    assert 2 <= p["stages"] <= 8 or p["stages"] == bpp
    assert p["stages"] * p["stage_bytes"] + 128 * rows * NT * 4 < p["smem_bytes"] <= 227 * 1024
    assert P == 1 or tiles <= 1024
    pre = -(-nbox * 256 // 2048)
    assert p["ws_bytes"] >= 4096 + 256 + M * pre * 4 + nbox * slice_bytes + (tiles * M * 512 if P > 1 else 0)


def check_rowdot_plan(p, M, K, N, sms):
    assert 2 <= M <= 8
    tiles = -(-N // 128)
    nbox = -(-K // 256)
    P, tpr = p["splits"], p["threads_per_row"]
    assert tpr in (2, 4, 8) and p["cols_per_thread"] == M
    assert p["ctas_per_split"] == tiles and p["grid"] == tiles * P
    bpp = -(-nbox // P)
    assert (P - 1) * bpp < nbox                                  # no empty piece
    assert M * bpp * 256 <= 48 * 1024                            # the piece's activation planes
    assert 1 <= p["stages"] <= min(8, bpp) and p["stage_bytes"] == 16384
    assert p["smem_bytes"] >= p["stages"] * 16384 + M * bpp * 256
    assert p["smem_bytes"] * max(1, 4 // tpr) <= 227 * 1024
    assert P == 1 or tiles <= 1024
    assert p["ws_bytes"] >= 4096 + 256 + M * nbox * 256 + (tiles * P * M * 512 if P > 1 else 0)


def test_kernel_routing():
    """Row-wise calls: 1 row on the dp4a GEMV, 2..3 rows on the
    row-per-thread kernel for matrices of at most 2 x SMs tiles, the tensor
    cores otherwise, except lm_head-sized matrices (at least 4 x SMs tiles in
    one K piece) at 2..4 rows: the warp-level kernel's persistent plan; an
    explicit qmma_max_m gives the warp-level kernel 2 rows up to it (any
    matrix), 1 switches it off; with the tensor cores switched off the
    row-per-thread kernel takes up to rowdot_max_m rows; the tuning moves
    every threshold."""
    try:
        route = lambda M, N=18944: w4.w4a8_plan_info(M, 3584, N, num_sms=152)["kernel"]
        assert [route(M) for M in (1, 2, 3, 4, 8, 9, 32, 64)] == [0, 2, 2, 1, 1, 1, 1, 1]
        assert [route(M, 152064) for M in (1, 2, 3, 4, 5, 8)] == [0, 3, 3, 3, 1, 1]   # lm_head: many tiles
        p = w4.w4a8_plan_info(4, 3584, 152064, num_sms=152)
        assert p["grid"] == 2 * 152 and p["splits"] == 1                 # two persistent CTAs per SM
        assert route(2, 77824 - 128) == 1 and route(2, 77824) == 3       # from 4 x 152 tiles
        w4.w4a8_set_tuning(qmma_max_m=1)
        assert [route(M, 152064) for M in (2, 3, 4)] == [1, 1, 1]         # switched off
        w4.w4a8_set_tuning()
        w4.w4a8_set_tuning(qmma_max_m=16)
        assert [route(M) for M in (2, 16, 17)] == [3, 3, 1]
        w4.w4a8_set_tuning(qmma_max_m=32, qmma_tiles_per_warp=1)
        assert w4.w4a8_plan_info(20, 3584, 18944, num_sms=152)["threads_per_row"] == 1
        w4.w4a8_set_tuning(qmma_max_m=32, qmma_tiles_per_warp=4, qmma_operands=1)  # binary16: 4 tiles a warp up to 32 rows
        assert [route(M) for M in (16, 17, 32)] == [3, 3, 3]
        p = w4.w4a8_plan_info(24, 3584, 18944, num_sms=152)
        check_qmma_plan(p, 24, 3584, 18944, 152, h16=True)
        w4.w4a8_set_tuning(qmma_max_m=32, qmma_tiles_per_warp=4)  # e4m3 (the default): up to 16 rows
        assert [route(M) for M in (16, 17)] == [3, 1]
        with pytest.raises(w4.W4A8Error):
            w4.w4a8_set_tuning(qmma_operands=3)
        with pytest.raises(w4.W4A8Error):
            w4.w4a8_set_tuning(qmma_tiles_per_warp=3)
        w4.w4a8_set_tuning(qmma_max_m=1, rowdot_max_m=8)
        assert [route(M) for M in (1, 2, 3, 8, 9, 64)] == [0, 2, 2, 2, 1, 1]
        assert route(8, 152064) == 2                                       # explicit: any matrix
        with pytest.raises(w4.W4A8Error):
            w4.w4a8_set_tuning(qmma_max_m=33)
        w4.w4a8_set_tuning(rowdot_max_m=4, qmma_max_m=1)
        assert [route(M) for M in (2, 4, 5)] == [2, 2, 1]
        w4.w4a8_set_tuning(rowdot_max_m=1, qmma_max_m=1)
        assert [route(M) for M in (2, 3)] == [1, 1]   # row-wise: the tensor cores from 2 rows
        w4.w4a8_set_tuning(rowdot_max_m=1, qmma_max_m=1, mma_min_m=3)
        assert [route(M) for M in (2, 3)] == [0, 1]
        for tpr in (2, 4, 8):
            w4.w4a8_set_tuning(force_threads_per_row=tpr, qmma_max_m=1, rowdot_max_m=8)
            p = w4.w4a8_plan_info(5, 3584, 18944, num_sms=152)
            assert p["threads_per_row"] == tpr and p["kernel"] == 2
            check_rowdot_plan(p, 5, 3584, 18944, 152)
        with pytest.raises(w4.W4A8Error):
            w4.w4a8_set_tuning(rowdot_max_m=9, qmma_max_m=1)
        with pytest.raises(w4.W4A8Error):
            w4.w4a8_set_tuning(mma_e4m3=3)
        w4.w4a8_set_tuning(mma_e4m3=2, rowdot_max_m=1, qmma_max_m=1)  # operand type does not change the plan
        assert w4.w4a8_plan_info(4, 3584, 18944, num_sms=152)["kernel"] == 1
        # group scales: the one-thread-per-row kernel at 1..8 rows, the tensor
        # cores above for groups of whole 128-code stages, else launches of 8 rows
        w4.w4a8_set_tuning()
        groute = lambda M, gs=128: w4.w4a8g_plan_info(M, 3584, 18944, gs, num_sms=152)
        assert [groute(M)["kernel"] for M in (1, 4, 8, 9, 64)] == [2, 2, 2, 1, 1]
        assert groute(4, 32)["kernel"] == 2 and groute(40, 32)["kernel"] == 2
        assert groute(40, 32)["cols_per_thread"] == 8 and groute(5)["cols_per_thread"] == 5
        w4.w4a8_set_tuning(rowdot_max_m=1, mma_min_m=65)
        assert groute(1)["kernel"] == 2 and groute(20)["cols_per_thread"] == 8
        w4.w4a8_set_tuning(mma_min_m=65, rowdot_max_m=1, qmma_max_m=1)
        assert w4.w4a8_plan_info(64, 3584, 18944, num_sms=152)["kernel"] == 0
        w4.w4a8_set_tuning(mma_min_m=2, rowdot_max_m=1, qmma_max_m=1)
        assert w4.w4a8_plan_info(2, 3584, 18944, num_sms=152)["kernel"] == 1
        assert w4.w4a8_plan_info(1, 3584, 18944, num_sms=152)["kernel"] == 0
        with pytest.raises(w4.W4A8Error):
            w4.w4a8_set_tuning(mma_min_m=1, qmma_max_m=1)
    finally:
        w4.w4a8_set_tuning(reset=True)


def test_forced_plans_respected():
    try:
        w4.w4a8_set_tuning(force_splits=4)
        assert w4.w4a8_plan_info(1, 3584, 3584, num_sms=152)["splits"] == 4
        w4.w4a8_set_tuning(force_threads_per_row=256)
        assert w4.w4a8_plan_info(1, 3584, 3584, num_sms=152)["threads_per_row"] == 256
        w4.w4a8_set_tuning(ring_bytes=8192)
        assert w4.w4a8_plan_info(1, 3584, 3584, num_sms=152)["stages"] == 2
    finally:
        w4.w4a8_set_tuning(reset=True)


# --------------------------------------------------------------------------
# group-wise scales
# --------------------------------------------------------------------------

def test_group_argument_checks(L):
    E_S, E_A, E_N = w4._binding.ERR_SHAPE, w4._binding.ERR_ALIGN, w4._binding.ERR_NULL
    for gs in (16, 48, 96, 3584, 0, -32, 8192):   # below 32, not a power of two, > K
        assert L.w4g_quantize_weights(P16, 4, 3584, gs, P16, P16, None) == E_S, gs
        assert L.w4a8g_linear(P16, 1, 3584, gs, P16, P16, 4, P16, None, None, None, 0, 0, None) == E_S, gs
        assert L.w4a8g_workspace_bytes(1, 3584, 4, gs) == 0
    assert L.w4g_quantize_weights(P16, 4, 3584, 1024, P16, P16, None) == E_S   # 1024 does not divide 3584
    assert L.w4g_quantize_weights(P16, 4, 3584, 128, P16, P16 + 4, None) == E_A  # scales 16-byte aligned
    assert L.w4g_quantize_weights(None, 4, 3584, 128, P16, P16, None) == E_N
    assert L.w4a8g_gemv(P16, P16, 1, 3584, 128, P16, P16 + 8, 4, P16, None, 0, 0, None) == E_A
    assert L.w4a8g_gemv(P16, None, 1, 3584, 128, P16, P16, 4, P16, None, 0, 0, None) == E_N
    assert L.w4a8g_gemv(P16, P16, 65, 3584, 128, P16, P16, 4, P16, None, 0, 0, None) == E_S
    assert L.w4a8g_linear(P16 + 8, 1, 3584, 128, P16, P16, 4, P16, None, None, None, 0, 0, None) == E_A
    arr = (ctypes.c_void_p * 2)(P16, P16)
    mis = (ctypes.c_void_p * 2)(P16, P16 + 4)
    ns = (ctypes.c_int64 * 2)(4, 4)
    assert L.w4a8g_linear_grouped(P16, 1, 3584, 128, 0, arr, arr, ns, arr, None, 0, 0, None) == E_S
    assert L.w4a8g_linear_grouped(P16, 1, 3584, 128, 2, arr, mis, ns, arr, None, 0, 0, None) == E_A


def test_group_scale_stride_matches_header():
    src = open(os.path.join(ROOT, "include", "w4a8.h")).read()
    assert "#define W4G_SCALE_STRIDE(K, group) ((((K) / (group)) + 3) / 4 * 4)" in src
    for K, gs, want in [(896, 128, 8), (3584, 128, 28), (18944, 128, 148), (4096, 4096, 4)]:
        assert w4.w4g_scale_stride(K, gs) == want


GROUP_SHAPES = [(1, 896, 512, 128), (1, 3584, 152064, 128), (1, 18944, 3584, 128),
                (1, 3584, 37888, 64), (2, 3584, 18944, 256), (8, 18944, 3584, 32), (1, 32, 7, 32),
                (3, 131072, 5, 1024), (1, 4096, 9, 4096), (8, 2048, 100, 512), (5, 8192, 40, 2048),
                (8, 131072, 2, 131072)]


def check_group_plan(p, M, K, N, gs, sms, splits=0):
    """The one-thread-per-row group kernel's plan: whole chunks per K piece,
    four CTAs of 128 threads per SM, and a workspace for the codes and the
    chunk sums of split tiles."""
    L = max(gs, 1024)
    nch = -(-K // L)
    nbox = -(-K // 256)
    tiles = -(-N // 128)
    P = p["splits"]
    assert p["kernel"] == 2 and p["threads_per_row"] in (1, 2, 4) and p["cols_per_thread"] == M
    assert p["chunks"] == nch and p["chunk_codes"] == L
    if splits:  # pieces of whole chunks: the requested count, or fewer when chunks do not divide
        want = -(-nch // -(-nch // min(splits, nch)))
        assert P == (want if tiles <= 1024 else 1)
    assert 1 <= P <= nch
    cpp = -(-nch // P)
    assert (P - 1) * cpp < nch                                   # no empty piece
    assert p["ctas_per_split"] == tiles and p["grid"] == tiles * P
    assert p["stage_bytes"] == 16384 and 1 <= p["stages"] <= 16
    assert p["smem_bytes"] >= p["stages"] * (16384 + M * 256)
    cps = min(4, -(-p["grid"] // sms))             # CTAs per SM the grid fills
    nph = p["threads_per_row"]                     # thread phases, each whole chunks of a piece
    assert p["smem_bytes"] * cps <= 227 * 1024
    assert p["stages"] * cps >= 12 or p["smem_bytes"] * cps > 227 * 1024 - (16384 + M * 256) * cps
    assert nph * cps <= 4 and nph <= cpp and (nph == 4 // cps or nph * 2 > cpp or nph == 1)
    if tiles >= sms and not splits:
        assert P == 1                              # every SM has a CTA already
    assert P == 1 or tiles <= 1024
    assert p["ws_bytes"] >= 4096 + 256 + M * nbox * 256 + (tiles * nch * M * 512 if P > 1 else 0)


@pytest.mark.parametrize("sms", [152, 148, 20, 1])
@pytest.mark.parametrize("splits", [0, 3, 7, 16])
def test_group_plans(sms, splits):
    """Every group-scale shape of 1..8 rows plans on the one-thread-per-row
    kernel, K pieces of whole fold chunks (a forced count is capped by the
    chunks), and the workspace query agrees with the plan."""
    try:
        w4.w4a8_set_tuning(force_splits=splits)
        for (M, K, N, gs) in GROUP_SHAPES:
            p = w4.w4a8g_plan_info(M, K, N, gs, num_sms=sms)
            check_group_plan(p, M, K, N, gs, sms, splits)
    finally:
        w4.w4a8_set_tuning(reset=True)


def test_group_workspace_covers_grouped_matrices():
    """A grouped group-scale call plans each matrix on its own inside the
    workspace sized for the total rows."""
    try:
        for splits in (0, 4):
            w4.w4a8_set_tuning(force_splits=splits)
            for sms in (152, 148, 20):
                for (M, K, gs) in [(1, 3584, 128), (8, 18944, 128), (3, 131072, 1024), (2, 896, 32)]:
                    full = w4.w4a8g_plan_info(M, K, 40000, gs, num_sms=sms)
                    for Np in (1, 7, 128, 129, 1000, 4608, 18944, 39999):
                        p = w4.w4a8g_plan_info(M, K, Np, gs, num_sms=sms)
                        check_group_plan(p, M, K, Np, gs, sms, splits)
                        assert p["ws_bytes"] <= full["ws_bytes"], (M, K, Np, sms)
    finally:
        w4.w4a8_set_tuning(reset=True)


# --------------------------------------------------------------------------
# IndexSoftmax host helpers and argument checks
# --------------------------------------------------------------------------

def test_isx_lut_and_c_int_match_oracle():
    import oracle
    o = oracle.load()
    for b, c in [(5, 6.6), (3, 5.5), (4, 7.7), (8, 5.5), (1, 2.0)]:
        assert w4.index_softmax_lut(b, c) == bytes(o.isx_lut(b, c)), (b, c)
    for c, d, sq, sk in [(6.6, 128, 4 / 127, 4 / 127), (2.5, 1, 1.0, 1.0), (6.6, 64, 0.01, 0.02),
                         (5.5, 128, 2.0 ** -5, 2.0 ** -5)]:
        assert w4.index_softmax_c_int(c, d, sq, sk) == o.isx_c_int(c, d, sq, sk)
    with pytest.raises(w4.W4A8Error):
        w4.index_softmax_c_int(6.6, 128, 1e-6, 1e-6)    # beyond 2^31 - 1
    with pytest.raises(w4.W4A8Error):
        w4.index_softmax_lut(9, 6.6)


def test_isx_argument_checks(L):
    E_S, E_A, E_N = w4._binding.ERR_SHAPE, w4._binding.ERR_ALIGN, w4._binding.ERR_NULL
    lut = (ctypes.c_uint8 * 32)(*w4.index_softmax_lut())
    zero_lut = (ctypes.c_uint8 * 32)()
    lp = ctypes.cast(lut, ctypes.c_void_p)
    assert L.index_softmax_u8(None, 1, 8, 100, 5, lp, P16, None) == E_N
    assert L.index_softmax_u8(P16, 1, 8, 100, 5, None, P16, None) == E_N
    assert L.index_softmax_u8(P16, 0, 8, 100, 5, lp, P16, None) == E_S
    assert L.index_softmax_u8(P16, 1, 0, 100, 5, lp, P16, None) == E_S
    assert L.index_softmax_u8(P16, 1, (1 << 23) + 1, 100, 5, lp, P16, None) == E_S
    assert L.index_softmax_u8(P16, 1, 8, -1, 5, lp, P16, None) == E_S
    assert L.index_softmax_u8(P16, 1, 8, 1 << 31, 5, lp, P16, None) == E_S
    assert L.index_softmax_u8(P16, 1, 8, 100, 0, lp, P16, None) == E_S
    assert L.index_softmax_u8(P16, 1, 8, 100, 9, lp, P16, None) == E_S
    assert L.index_softmax_u8(P16, 1, 8, 100, 5, ctypes.cast(zero_lut, ctypes.c_void_p), P16, None) == E_S
    assert L.index_softmax_u8(P16 + 2, 1, 8, 100, 5, lp, P16, None) == E_A


def test_group_tensor_core_plans():
    """Group scales with 3..64 rows take the tensor cores when the group is a
    whole number of 128-code stages (at most 16384 codes); K pieces hold
    whole fold chunks, and a split plan's workspace holds one fp32 sum per
    output and chunk (at most 32 MB); other groups run launches of up to 8
    rows on the one-thread-per-row kernel."""
    try:
        w4.w4a8_set_tuning(rowdot_max_m=1, qmma_max_m=1)  # 1..8 rows would take the one-thread-per-row kernel
        for sms in (152, 148, 20):
            for (M, K, N, gs) in [(3, 3584, 300, 128), (16, 3584, 18944, 128), (64, 18944, 3584, 128),
                                  (4, 3584, 1000, 256), (8, 2048, 200, 512), (33, 896, 100, 128),
                                  (5, 32768, 64, 16384), (40, 3072, 130, 1024)]:
                p = w4.w4a8g_plan_info(M, K, N, gs, num_sms=sms)
                assert p["kernel"] == 1, (M, K, N, gs)
                L = max(gs, 1024)
                nch, tiles, P = -(-K // L), -(-N // 128), p["splits"]
                assert p["chunks"] == nch and p["chunk_codes"] == L
                assert 1 <= P <= nch and p["grid"] == tiles * P and p["ctas_per_split"] == tiles
                cpp = -(-nch // P)                        # whole chunks per piece, none empty
                assert (P - 1) * cpp < nch
                part = tiles * nch * M * 512 if P > 1 else 0
                assert part <= 32 << 20
                assert p["ws_bytes"] >= 4096 + 256 + M * K * 2 + part
                if tiles * 5 >= 2 * sms * 4 or nch == 1:
                    assert P == 1
            for (M, K, N, gs) in [(3, 1024, 77, 32), (8, 3584, 100, 64), (20, 3584, 100, 64)]:
                p = w4.w4a8g_plan_info(M, K, N, gs, num_sms=sms)
                assert p["kernel"] == 2 and p["cols_per_thread"] == min(M, 8)
        w4.w4a8_set_tuning(mma_min_m=65, rowdot_max_m=1, qmma_max_m=1)
        assert w4.w4a8g_plan_info(16, 3584, 18944, 128, num_sms=152)["kernel"] == 2
    finally:
        w4.w4a8_set_tuning(reset=True)


def test_rowdot_workspace_covers_grouped_matrices():
    """A grouped call plans each matrix on its own inside the workspace sized
    for the total rows: every smaller matrix's plan needs no more, and plans
    that never split K do not reserve partial sums per tile."""
    try:
        w4.w4a8_set_tuning(qmma_max_m=1, rowdot_max_m=8)
        for sms in (152, 148, 20):
            for (M, K) in [(2, 3584), (8, 3584), (8, 18944), (5, 131072), (3, 896)]:
                N = 40000
                full = w4.w4a8_plan_info(M, K, N, num_sms=sms)
                assert full["kernel"] == 2
                for Np in (1, 7, 128, 129, 1000, 4608, 18944, 39999):
                    p = w4.w4a8_plan_info(M, K, Np, num_sms=sms)
                    check_rowdot_plan(p, M, K, Np, sms)
                    assert p["ws_bytes"] <= full["ws_bytes"], (M, K, Np, sms)
        p = w4.w4a8_plan_info(8, 3584, 152064, num_sms=152)  # lm_head: one piece per tile
        assert p["splits"] == 1 and p["ws_bytes"] < 2 * 1024 * 1024
    finally:
        w4.w4a8_set_tuning(reset=True)


def test_mma_workspace_covers_grouped_matrices():
    """The same for the tensor-core kernel: each matrix of a grouped call
    (its own plan, its own K split) fits the workspace planned for the total
    rows, with or without a forced split count."""
    try:
        for splits in (0, 3):
            w4.w4a8_set_tuning(force_splits=splits, qmma_max_m=1)
            for sms in (152, 148, 20):
                for (M, K) in [(4, 3584), (16, 3584), (64, 18944), (9, 131072), (33, 896)]:
                    N = 40000
                    full = w4.w4a8_plan_info(M, K, N, num_sms=sms)
                    assert full["kernel"] == 1
                    for Np in (1, 7, 128, 129, 1000, 4608, 18944, 39999):
                        p = w4.w4a8_plan_info(M, K, Np, num_sms=sms)
                        if p["kernel"] != 1:
                            continue
                        check_mma_plan(p, M, K, Np, sms)
                        assert p["ws_bytes"] <= full["ws_bytes"], (M, K, Np, sms)
    finally:
        w4.w4a8_set_tuning(reset=True)


def test_qmma_workspace_covers_grouped_matrices():
    """The same for the warp-level MMA kernel: each matrix of a grouped call
    fits the workspace planned for the total rows."""
    try:
        w4.w4a8_set_tuning(qmma_max_m=32)
        _qmma_grouped_cases()
    finally:
        w4.w4a8_set_tuning(reset=True)


def _qmma_grouped_cases():
    for sms in (152, 148, 20):
        for (M, K) in [(2, 3584), (8, 3584), (16, 18944), (32, 131072), (3, 896), (32, 3584)]:
            N = 40000
            full = w4.w4a8_plan_info(M, K, N, num_sms=sms)
            assert full["kernel"] == 3
            for Np in (1, 7, 128, 129, 1000, 4608, 18944, 39999):
                p = w4.w4a8_plan_info(M, K, Np, num_sms=sms)
                check_qmma_plan(p, M, K, Np, sms)
                assert p["ws_bytes"] <= full["ws_bytes"], (M, K, Np, sms)


def test_qmma_binary16_plans():
    """Warp-level MMA plans with binary16 operands (qmma_operands = 1) for
    every shape of the plan table: n-tiles of 8 rows, 4096-byte slices per
    n-tile, at most 64 boxes (16384 codes) per warp accumulator."""
    try:
        w4.w4a8_set_tuning(qmma_max_m=32, qmma_operands=1)
        for sms in (152, 20):
            for (M, K, N) in SHAPES + [(7, 131072, 300), (12, 65536, 2000), (32, 512, 200000)]:
                if not 2 <= M <= 32:
                    continue
                p = w4.w4a8_plan_info(M, K, N, num_sms=sms)
                assert p["kernel"] == 3
                check_qmma_plan(p, M, K, N, sms, h16=True)
    finally:
        w4.w4a8_set_tuning(reset=True)
