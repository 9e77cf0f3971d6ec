"""ctypes binding of libw4a8.so: the entry points of include/w4a8.h under the
same names, taking torch CUDA tensors.

Argument marshalling only: every step of the linear runs in the library's
CUDA kernels.  There is no fallback: if the library is missing or a call is
rejected, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libw4a8.so")

OK = 0
ERR_NULL, ERR_ALIGN, ERR_SHAPE, ERR_WORKSPACE, ERR_CUDA = 1, 2, 3, 4, 5
LAUNCH_PDL = 1
W4A8_MAX_M = 64
W8A16_MAX_M = 64

EXPORTS = [
    "w4_quantize_weights", "w8_quantize_weights", "act_quantize_i8",
    "w4a8_workspace_bytes", "w4a8_gemv", "w4a8_linear",
    "w8a16_workspace_bytes", "w8a16_gemv",
    "w4a8_last_error", "w4a8_device_error", "w4a8_set_tuning", "w4a8_plan_info",
    "w4a8_linear_noalloc", "w4a8_linear_grouped", "w4a8_linear_prefetch", "w4a8_linear_grouped_prefetch",
    "w4g_quantize_weights", "w4a8g_workspace_bytes", "w4a8g_gemv", "w4a8g_linear",
    "w4a8g_linear_grouped", "w4a8g_plan_info",
    "index_softmax_lut", "index_softmax_c_int", "index_softmax_u8",
    "w4_interleave_rows", "w4a8_gate_up_silu_workspace_bytes", "w4a8_gate_up_silu", "w4a8_silu_mul",
]


class W4A8Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("status %d: %s" % (status, message))
        self.status = status


class _Tuning(ctypes.Structure):
    _fields_ = [("force_splits", ctypes.c_int), ("force_threads_per_row", ctypes.c_int),
                ("ring_bytes", ctypes.c_int), ("ctas_per_sm", ctypes.c_int),
                ("mma_min_m", ctypes.c_int), ("rowdot_max_m", ctypes.c_int),
                ("mma_e4m3", ctypes.c_int), ("qmma_max_m", ctypes.c_int),
                ("qmma_tiles_per_warp", ctypes.c_int), ("stall_test_us", ctypes.c_int),
                ("qmma_operands", ctypes.c_int)]


_i64, _p, _u = ctypes.c_int64, ctypes.c_void_p, ctypes.c_uint
_SIGS = {
    "w4_quantize_weights": (ctypes.c_int, [_p, _i64, _i64, _p, _p, _p]),
    "w8_quantize_weights": (ctypes.c_int, [_p, _i64, _i64, _p, _p, _p]),
    "act_quantize_i8": (ctypes.c_int, [_p, _i64, _i64, _p, _p, _p]),
    "w4a8_workspace_bytes": (ctypes.c_size_t, [_i64, _i64, _i64]),
    "w4a8_gemv": (ctypes.c_int, [_p, _p, _i64, _i64, _p, _p, _i64, _p, _p, _p, ctypes.c_size_t, _u, _p]),
    "w4a8_linear": (ctypes.c_int, [_p, _i64, _i64, _p, _p, _i64, _p, _p, _p, _p, _p, ctypes.c_size_t, _u, _p]),
    "w4a8_linear_prefetch": (ctypes.c_int, [_p, _i64, _i64, _p, _p, _i64, _p, _p, ctypes.c_size_t, _u, _p, _p,
                                            ctypes.c_size_t]),
    "w4a8_linear_grouped_prefetch": (ctypes.c_int, [_p, _i64, _i64, ctypes.c_int, _p, _p, _p, _p, _p,
                                                    ctypes.c_size_t, _u, _p, _p, ctypes.c_size_t]),
    "w4a8_linear_noalloc": (ctypes.c_int, [_p, _i64, _i64, _p, _p, _i64, _p, _u, _p]),
    "w4a8_linear_grouped": (ctypes.c_int, [_p, _i64, _i64, ctypes.c_int, _p, _p, _p, _p, _p,
                                           ctypes.c_size_t, _u, _p]),
    "w8a16_workspace_bytes": (ctypes.c_size_t, [_i64, _i64, _i64]),
    "w8a16_gemv": (ctypes.c_int, [_p, _i64, _i64, _p, _p, _i64, _p, _p, ctypes.c_size_t, _u, _p]),
    "w4a8_last_error": (ctypes.c_char_p, []),
    "w4a8_device_error": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint), _p]),
    "w4a8_set_tuning": (ctypes.c_int, [ctypes.POINTER(_Tuning)]),
    "w4a8_plan_info": (ctypes.c_int, [_i64, _i64, _i64, ctypes.c_int, ctypes.c_int,
                                      ctypes.POINTER(ctypes.c_int), ctypes.c_int]),
    "w4g_quantize_weights": (ctypes.c_int, [_p, _i64, _i64, _i64, _p, _p, _p]),
    "w4a8g_workspace_bytes": (ctypes.c_size_t, [_i64, _i64, _i64, _i64]),
    "w4a8g_gemv": (ctypes.c_int, [_p, _p, _i64, _i64, _i64, _p, _p, _i64, _p, _p, ctypes.c_size_t,
                                  _u, _p]),
    "w4a8g_linear": (ctypes.c_int, [_p, _i64, _i64, _i64, _p, _p, _i64, _p, _p, _p, _p,
                                    ctypes.c_size_t, _u, _p]),
    "w4a8g_linear_grouped": (ctypes.c_int, [_p, _i64, _i64, _i64, ctypes.c_int, _p, _p, _p, _p,
                                            _p, ctypes.c_size_t, _u, _p]),
    "w4a8g_plan_info": (ctypes.c_int, [_i64, _i64, _i64, _i64, ctypes.c_int,
                                       ctypes.POINTER(ctypes.c_int), ctypes.c_int]),
    "index_softmax_lut": (ctypes.c_int, [ctypes.c_int, ctypes.c_double, _p]),
    "index_softmax_c_int": (_i64, [ctypes.c_double, _i64, ctypes.c_float, ctypes.c_float]),
    "index_softmax_u8": (ctypes.c_int, [_p, _i64, _i64, _i64, ctypes.c_int, _p, _p, _p]),
    "w4_interleave_rows": (ctypes.c_int, [_p, _p, _p, _p, _i64, _i64, _p, _p, _p]),
    "w4a8_gate_up_silu_workspace_bytes": (ctypes.c_size_t, [_i64, _i64, _i64]),
    "w4a8_gate_up_silu": (ctypes.c_int, [_p, _i64, _i64, _p, _p, _i64, _p, _p, _p, ctypes.c_size_t, _u, _p]),
    "w4a8_silu_mul": (ctypes.c_int, [_p, _p, _i64, _i64, _p, _u, _p]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libw4a8.so not built: call __graft_entry__.build() or "
                              "python -m bit_weight_quantized_w4a8_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(st: int):
    if st != OK:
        raise W4A8Error(st, lib().w4a8_last_error().decode(errors="replace"))


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _want(t, dtype, name, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))


_ws_cache = {}


def _workspace(nbytes: int, device: torch.device, ws):
    """Caller-provided workspace, or a cached zero-filled one per device."""
    if nbytes == 0:
        return ws
    if ws is not None:
        return ws
    key = device.index if device.index is not None else torch.cuda.current_device()
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.zeros(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


# --------------------------------------------------------------------------
# entry points
# --------------------------------------------------------------------------

def w4_quantize_weights(W: torch.Tensor, Wq=None, sw=None):
    """W [N][K] fp32 -> (Wq [N][K/2] uint8, sw [N] fp32)."""
    _want(W, torch.float32, "W")
    N, K = W.shape
    Wq = torch.empty((N, K // 2), dtype=torch.uint8, device=W.device) if Wq is None else Wq
    sw = torch.empty((N,), dtype=torch.float32, device=W.device) if sw is None else sw
    _want(Wq, torch.uint8, "Wq", (N, K // 2))
    _want(sw, torch.float32, "sw", (N,))
    _check(lib().w4_quantize_weights(_ptr(W), N, K, _ptr(Wq), _ptr(sw), _stream(W)))
    return Wq, sw


def w8_quantize_weights(W: torch.Tensor, Wq8=None, sw16=None):
    """W [N][K] fp32 -> (Wq8 [N][K] int8, sw16 [N] fp16)."""
    _want(W, torch.float32, "W")
    N, K = W.shape
    Wq8 = torch.empty((N, K), dtype=torch.int8, device=W.device) if Wq8 is None else Wq8
    sw16 = torch.empty((N,), dtype=torch.float16, device=W.device) if sw16 is None else sw16
    _want(Wq8, torch.int8, "Wq8", (N, K))
    _want(sw16, torch.float16, "sw16", (N,))
    _check(lib().w8_quantize_weights(_ptr(W), N, K, _ptr(Wq8), _ptr(sw16), _stream(W)))
    return Wq8, sw16


def act_quantize_i8(X: torch.Tensor, Xq=None, sa=None):
    """X [M][K] fp16 -> (Xq [M][K] int8, sa [M] fp32)."""
    _want(X, torch.float16, "X")
    M, K = X.shape
    Xq = torch.empty((M, K), dtype=torch.int8, device=X.device) if Xq is None else Xq
    sa = torch.empty((M,), dtype=torch.float32, device=X.device) if sa is None else sa
    _want(Xq, torch.int8, "Xq", (M, K))
    _want(sa, torch.float32, "sa", (M,))
    _check(lib().act_quantize_i8(_ptr(X), M, K, _ptr(Xq), _ptr(sa), _stream(X)))
    return Xq, sa


def w4a8_workspace_bytes(M: int, K: int, N: int) -> int:
    return int(lib().w4a8_workspace_bytes(M, K, N))


def w8a16_workspace_bytes(M: int, K: int, N: int) -> int:
    return int(lib().w8a16_workspace_bytes(M, K, N))


def w4a8_gemv(Xq, sa, Wq, sw, Y=None, acc_out=None, ws=None, flags: int = 0):
    """Y[m][n] = ((float)sum_k Xq[m,k] q[n,k] * sw[n]) * sa[m]; returns Y."""
    _want(Xq, torch.int8, "Xq")
    M, K = Xq.shape
    N = Wq.shape[0]
    _want(sa, torch.float32, "sa", (M,))
    _want(Wq, torch.uint8, "Wq", (N, K // 2))
    _want(sw, torch.float32, "sw", (N,))
    Y = torch.empty((M, N), dtype=torch.float32, device=Xq.device) if Y is None else Y
    _want(Y, torch.float32, "Y", (M, N))
    if acc_out is not None:
        _want(acc_out, torch.int32, "acc_out", (M, N))
    nbytes = w4a8_workspace_bytes(M, K, N)
    ws = _workspace(nbytes, Xq.device, ws)
    _check(lib().w4a8_gemv(_ptr(Xq), _ptr(sa), M, K, _ptr(Wq), _ptr(sw), N, _ptr(Y), _ptr(acc_out),
                           _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(), flags,
                           _stream(Xq)))
    return Y


def _prefetch_arg(prefetch, prefetch_bytes):
    if prefetch is None:
        return None, 0
    if not isinstance(prefetch, torch.Tensor) or not prefetch.is_cuda:
        raise TypeError("prefetch must be a CUDA tensor")
    nb = prefetch.numel() * prefetch.element_size()
    return prefetch.data_ptr(), min(nb, int(prefetch_bytes) if prefetch_bytes else nb)


def w4a8_linear(X, Wq, sw, Y=None, Xq_out=None, sa_out=None, acc_out=None, ws=None,
                flags: int = 0, prefetch=None, prefetch_bytes: int = 0):
    """Fused activation quantization + W4A8 product; returns Y.  `prefetch`
    (a CUDA tensor, e.g. the next launch's packed weights) and
    `prefetch_bytes` (0 = all of it): an L2 prefetch hint for the next
    launch (w4a8_linear_prefetch; the optional outputs are then not taken)."""
    _want(X, torch.float16, "X")
    M, K = X.shape
    N = Wq.shape[0]
    _want(Wq, torch.uint8, "Wq", (N, K // 2))
    _want(sw, torch.float32, "sw", (N,))
    Y = torch.empty((M, N), dtype=torch.float32, device=X.device) if Y is None else Y
    _want(Y, torch.float32, "Y", (M, N))
    if Xq_out is not None:
        _want(Xq_out, torch.int8, "Xq_out", (M, K))
    if sa_out is not None:
        _want(sa_out, torch.float32, "sa_out", (M,))
    if acc_out is not None:
        _want(acc_out, torch.int32, "acc_out", (M, N))
    nbytes = w4a8_workspace_bytes(M, K, N)
    ws = _workspace(nbytes, X.device, ws)
    wsb = 0 if ws is None else ws.numel() * ws.element_size()
    if prefetch is not None:
        if Xq_out is not None or sa_out is not None or acc_out is not None:
            raise ValueError("the prefetching call takes no optional outputs")
        pp, pb = _prefetch_arg(prefetch, prefetch_bytes)
        _check(lib().w4a8_linear_prefetch(_ptr(X), M, K, _ptr(Wq), _ptr(sw), N, _ptr(Y), _ptr(ws), wsb,
                                          flags, _stream(X), pp, pb))
        return Y
    _check(lib().w4a8_linear(_ptr(X), M, K, _ptr(Wq), _ptr(sw), N, _ptr(Y), _ptr(Xq_out),
                             _ptr(sa_out), _ptr(acc_out), _ptr(ws), wsb, flags, _stream(X)))
    return Y


def w4a8_linear_grouped(X, Wqs, sws, Ys=None, ws=None, flags: int = 0, prefetch=None,
                        prefetch_bytes: int = 0):
    """One launch for several weight matrices sharing X (e.g. q/k/v); returns
    the list of outputs, each bit-identical to w4a8_linear on its own.
    `prefetch`, `prefetch_bytes`: as in w4a8_linear."""
    _want(X, torch.float16, "X")
    M, K = X.shape
    G = len(Wqs)
    if G != len(sws) or not 1 <= G <= 4:
        raise ValueError("need 1..4 weight matrices with one scale vector each")
    Ns = [int(w.shape[0]) for w in Wqs]
    for g in range(G):
        _want(Wqs[g], torch.uint8, "Wq[%d]" % g, (Ns[g], K // 2))
        _want(sws[g], torch.float32, "sw[%d]" % g, (Ns[g],))
    if Ys is None:
        Ys = [torch.empty((M, n), dtype=torch.float32, device=X.device) for n in Ns]
    for g in range(G):
        _want(Ys[g], torch.float32, "Y[%d]" % g, (M, Ns[g]))
    arr_p = ctypes.c_void_p * G
    wq_a = arr_p(*[w.data_ptr() for w in Wqs])
    sw_a = arr_p(*[s.data_ptr() for s in sws])
    y_a = arr_p(*[y.data_ptr() for y in Ys])
    n_a = (ctypes.c_int64 * G)(*Ns)
    nbytes = w4a8_workspace_bytes(M, K, sum(Ns))
    ws = _workspace(nbytes, X.device, ws)
    wsb = 0 if ws is None else ws.numel() * ws.element_size()
    args = (_ptr(X), M, K, G, ctypes.cast(wq_a, ctypes.c_void_p), ctypes.cast(sw_a, ctypes.c_void_p),
            ctypes.cast(n_a, ctypes.c_void_p), ctypes.cast(y_a, ctypes.c_void_p), _ptr(ws), wsb, flags,
            _stream(X))
    if prefetch is not None:
        pp, pb = _prefetch_arg(prefetch, prefetch_bytes)
        _check(lib().w4a8_linear_grouped_prefetch(*args, pp, pb))
    else:
        _check(lib().w4a8_linear_grouped(*args))
    return Ys


def w4a8_linear_noalloc(X, Wq, sw, Y=None, flags: int = 0):
    """w4a8_linear for callers that cannot provide workspace memory: the
    split-K scratch is the library's static per-GPU array (see the C header
    for its limit and for why calls overlapping on the GPU must be avoided).
    Allocates nothing when Y is given."""
    _want(X, torch.float16, "X")
    M, K = X.shape
    N = Wq.shape[0]
    _want(Wq, torch.uint8, "Wq", (N, K // 2))
    _want(sw, torch.float32, "sw", (N,))
    Y = torch.empty((M, N), dtype=torch.float32, device=X.device) if Y is None else Y
    _want(Y, torch.float32, "Y", (M, N))
    _check(lib().w4a8_linear_noalloc(_ptr(X), M, K, _ptr(Wq), _ptr(sw), N, _ptr(Y), flags,
                                     _stream(X)))
    return Y


def w8a16_gemv(X, Wq8, sw16, Y=None, ws=None, flags: int = 0):
    """Y[m][n] = float(sw16[n]) * sum_k q[n,k] * x[m,k]; returns Y."""
    _want(X, torch.float16, "X")
    M, K = X.shape
    N = Wq8.shape[0]
    _want(Wq8, torch.int8, "Wq8", (N, K))
    _want(sw16, torch.float16, "sw16", (N,))
    Y = torch.empty((M, N), dtype=torch.float32, device=X.device) if Y is None else Y
    _want(Y, torch.float32, "Y", (M, N))
    nbytes = w8a16_workspace_bytes(M, K, N)
    ws = _workspace(nbytes, X.device, ws)
    _check(lib().w8a16_gemv(_ptr(X), M, K, _ptr(Wq8), _ptr(sw16), N, _ptr(Y), _ptr(ws),
                            0 if ws is None else ws.numel() * ws.element_size(), flags,
                            _stream(X)))
    return Y


# -- the MLP's gated product ---------------------------------------------------

def w4_interleave_rows(Wq_a, sw_a, Wq_b, sw_b, Wq_out=None, sw_out=None):
    """Rows of two packed matrices interleaved: (Wq [2N][K/2], sw [2N])."""
    N, half = Wq_a.shape
    for t, dt, nm, shp in ((Wq_a, torch.uint8, "Wq_a", (N, half)), (Wq_b, torch.uint8, "Wq_b", (N, half)),
                           (sw_a, torch.float32, "sw_a", (N,)), (sw_b, torch.float32, "sw_b", (N,))):
        _want(t, dt, nm, shp)
    Wq_out = torch.empty((2 * N, half), dtype=torch.uint8, device=Wq_a.device) if Wq_out is None else Wq_out
    sw_out = torch.empty((2 * N,), dtype=torch.float32, device=Wq_a.device) if sw_out is None else sw_out
    _want(Wq_out, torch.uint8, "Wq_out", (2 * N, half))
    _want(sw_out, torch.float32, "sw_out", (2 * N,))
    _check(lib().w4_interleave_rows(_ptr(Wq_a), _ptr(sw_a), _ptr(Wq_b), _ptr(sw_b), N, 2 * half,
                                    _ptr(Wq_out), _ptr(sw_out), _stream(Wq_a)))
    return Wq_out, sw_out


def w4a8_gate_up_silu_workspace_bytes(M: int, K: int, N: int) -> int:
    return int(lib().w4a8_gate_up_silu_workspace_bytes(M, K, N))


def w4a8_gate_up_silu(X, Wq_gu, sw_gu, H=None, Y_gu=None, ws=None, flags: int = 0):
    """Gate/up projections of interleaved weights with the gated product in
    the epilogue; returns (H [M][N] fp16, Y_gu [M][2N] fp32)."""
    _want(X, torch.float16, "X")
    M, K = X.shape
    N2 = Wq_gu.shape[0]
    if N2 % 2:
        raise ValueError("Wq_gu must have an even number of rows (gate/up pairs)")
    N = N2 // 2
    _want(Wq_gu, torch.uint8, "Wq_gu", (N2, K // 2))
    _want(sw_gu, torch.float32, "sw_gu", (N2,))
    H = torch.empty((M, N), dtype=torch.float16, device=X.device) if H is None else H
    Y_gu = torch.empty((M, N2), dtype=torch.float32, device=X.device) if Y_gu is None else Y_gu
    _want(H, torch.float16, "H", (M, N))
    _want(Y_gu, torch.float32, "Y_gu", (M, N2))
    ws = _workspace(w4a8_gate_up_silu_workspace_bytes(M, K, N), X.device, ws)
    _check(lib().w4a8_gate_up_silu(_ptr(X), M, K, _ptr(Wq_gu), _ptr(sw_gu), N, _ptr(Y_gu), _ptr(H), _ptr(ws),
                                   0 if ws is None else ws.numel() * ws.element_size(), flags, _stream(X)))
    return H, Y_gu


def w4a8_silu_mul(g, u, H=None, flags: int = 0):
    """H = fp16(silu(g) * u), g and u [M][N] fp32; returns H."""
    _want(g, torch.float32, "g")
    M, N = g.shape
    _want(u, torch.float32, "u", (M, N))
    H = torch.empty((M, N), dtype=torch.float16, device=g.device) if H is None else H
    _want(H, torch.float16, "H", (M, N))
    _check(lib().w4a8_silu_mul(_ptr(g), _ptr(u), M, N, _ptr(H), flags, _stream(g)))
    return H


# -- group-wise INT4 scales -------------------------------------------------

def w4g_scale_stride(K: int, group: int) -> int:
    """Floats per row of the group-scale matrix: K/group rounded up to a
    multiple of 4 (the W4G_SCALE_STRIDE layout of the C header)."""
    return (K // group + 3) // 4 * 4


def w4g_quantize_weights(W: torch.Tensor, group: int, Wq=None, sg=None):
    """W [N][K] fp32 -> (Wq [N][K/2] uint8, sg [N][stride] fp32)."""
    _want(W, torch.float32, "W")
    N, K = W.shape
    ld = w4g_scale_stride(K, group) if group > 0 else 0
    Wq = torch.empty((N, K // 2), dtype=torch.uint8, device=W.device) if Wq is None else Wq
    sg = torch.empty((N, ld), dtype=torch.float32, device=W.device) if sg is None else sg
    _want(Wq, torch.uint8, "Wq", (N, K // 2))
    _want(sg, torch.float32, "sg", (N, ld))
    _check(lib().w4g_quantize_weights(_ptr(W), N, K, group, _ptr(Wq), _ptr(sg), _stream(W)))
    return Wq, sg


def w4a8g_workspace_bytes(M: int, K: int, N: int, group: int) -> int:
    return int(lib().w4a8g_workspace_bytes(M, K, N, group))


def _want_group(Wq, sg, N, K, group, name=""):
    _want(Wq, torch.uint8, "Wq" + name, (N, K // 2))
    _want(sg, torch.float32, "sg" + name, (N, w4g_scale_stride(K, group) if group > 0 else 0))


def w4a8g_gemv(Xq, sa, Wq, sg, group: int, Y=None, ws=None, flags: int = 0):
    """Y[m][n] = sa[m] * sum_g sg[n][g] * acc_g[m][n] (group-wise scales); returns Y."""
    _want(Xq, torch.int8, "Xq")
    M, K = Xq.shape
    N = Wq.shape[0]
    _want(sa, torch.float32, "sa", (M,))
    _want_group(Wq, sg, N, K, group)
    Y = torch.empty((M, N), dtype=torch.float32, device=Xq.device) if Y is None else Y
    _want(Y, torch.float32, "Y", (M, N))
    ws = _workspace(w4a8g_workspace_bytes(M, K, N, group), Xq.device, ws)
    _check(lib().w4a8g_gemv(_ptr(Xq), _ptr(sa), M, K, group, _ptr(Wq), _ptr(sg), N, _ptr(Y),
                            _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(), flags,
                            _stream(Xq)))
    return Y


def w4a8g_linear(X, Wq, sg, group: int, Y=None, Xq_out=None, sa_out=None, ws=None,
                 flags: int = 0):
    """Fused activation quantization + group-scale W4A8 product; returns Y."""
    _want(X, torch.float16, "X")
    M, K = X.shape
    N = Wq.shape[0]
    _want_group(Wq, sg, N, K, group)
    Y = torch.empty((M, N), dtype=torch.float32, device=X.device) if Y is None else Y
    _want(Y, torch.float32, "Y", (M, N))
    if Xq_out is not None:
        _want(Xq_out, torch.int8, "Xq_out", (M, K))
    if sa_out is not None:
        _want(sa_out, torch.float32, "sa_out", (M,))
    ws = _workspace(w4a8g_workspace_bytes(M, K, N, group), X.device, ws)
    _check(lib().w4a8g_linear(_ptr(X), M, K, group, _ptr(Wq), _ptr(sg), N, _ptr(Y),
                              _ptr(Xq_out), _ptr(sa_out), _ptr(ws),
                              0 if ws is None else ws.numel() * ws.element_size(), flags,
                              _stream(X)))
    return Y


def w4a8g_linear_grouped(X, Wqs, sgs, group: int, Ys=None, ws=None, flags: int = 0):
    """One launch for several group-scale weight matrices sharing X; returns
    the list of outputs."""
    _want(X, torch.float16, "X")
    M, K = X.shape
    G = len(Wqs)
    if G != len(sgs) or not 1 <= G <= 4:
        raise ValueError("need 1..4 weight matrices with one scale matrix each")
    Ns = [int(w.shape[0]) for w in Wqs]
    for g in range(G):
        _want_group(Wqs[g], sgs[g], Ns[g], K, group, "[%d]" % g)
    if Ys is None:
        Ys = [torch.empty((M, n), dtype=torch.float32, device=X.device) for n in Ns]
    for g in range(G):
        _want(Ys[g], torch.float32, "Y[%d]" % g, (M, Ns[g]))
    arr_p = ctypes.c_void_p * G
    wq_a = arr_p(*[w.data_ptr() for w in Wqs])
    sg_a = arr_p(*[t.data_ptr() for t in sgs])
    y_a = arr_p(*[y.data_ptr() for y in Ys])
    n_a = (ctypes.c_int64 * G)(*Ns)
    ws = _workspace(w4a8g_workspace_bytes(M, K, sum(Ns), group), X.device, ws)
    _check(lib().w4a8g_linear_grouped(_ptr(X), M, K, group, G, ctypes.cast(wq_a, ctypes.c_void_p),
                                      ctypes.cast(sg_a, ctypes.c_void_p),
                                      ctypes.cast(n_a, ctypes.c_void_p),
                                      ctypes.cast(y_a, ctypes.c_void_p), _ptr(ws),
                                      0 if ws is None else ws.numel() * ws.element_size(), flags,
                                      _stream(X)))
    return Ys


# -- IndexSoftmax -------------------------------------------------------------

ISX_DEFAULT_B = 5
ISX_DEFAULT_C = 6.6


def index_softmax_lut(b: int = ISX_DEFAULT_B, c: float = ISX_DEFAULT_C) -> bytes:
    """The 2^b-entry UINT8 exponent table (computed on the host)."""
    buf = (ctypes.c_uint8 * (1 << b))() if 1 <= b <= 8 else (ctypes.c_uint8 * 1)()
    _check(lib().index_softmax_lut(b, c, ctypes.cast(buf, ctypes.c_void_p)))
    return bytes(buf)


def index_softmax_c_int(c: float, d: int, s_q: float, s_k: float) -> int:
    v = int(lib().index_softmax_c_int(c, d, s_q, s_k))
    if v < 0:
        raise W4A8Error(ERR_SHAPE, "index_softmax_c_int: arguments out of range")
    return v


def index_softmax_u8(A, c_int: int, b: int = ISX_DEFAULT_B, lut: bytes = None, P=None):
    """int32 logits [rows][cols] (CUDA) -> UINT8 probabilities; returns P."""
    _want(A, torch.int32, "A")
    rows, cols = A.shape
    P = torch.empty((rows, cols), dtype=torch.uint8, device=A.device) if P is None else P
    _want(P, torch.uint8, "P", (rows, cols))
    lut = index_softmax_lut(b) if lut is None else bytes(lut)
    if len(lut) != (1 << b):
        raise ValueError("lut must have 2^b entries")
    lut_buf = (ctypes.c_uint8 * len(lut)).from_buffer_copy(lut)
    _check(lib().index_softmax_u8(_ptr(A), rows, cols, c_int, b,
                                  ctypes.cast(lut_buf, ctypes.c_void_p), _ptr(P), _stream(A)))
    return P


def w4a8_last_error() -> str:
    return lib().w4a8_last_error().decode(errors="replace")


def w4a8_device_error(device=None) -> int:
    """Reads and clears the device error word (synchronises the current stream)."""
    flags = ctypes.c_uint(0)
    stream = torch.cuda.current_stream(device).cuda_stream
    _check(lib().w4a8_device_error(ctypes.byref(flags), stream))
    return int(flags.value)


def w4a8_set_tuning(force_splits: int = 0, force_threads_per_row: int = 0,
                    ring_bytes: int = 0, ctas_per_sm: int = 0, mma_min_m: int = 0,
                    rowdot_max_m: int = 0, mma_e4m3: int = 0, qmma_max_m: int = 0,
                    qmma_tiles_per_warp: int = 0, stall_test_us: int = 0, qmma_operands: int = 0,
                    reset: bool = False):
    if reset:
        _check(lib().w4a8_set_tuning(None))
        return
    t = _Tuning(force_splits, force_threads_per_row, ring_bytes, ctas_per_sm, mma_min_m,
                rowdot_max_m, mma_e4m3, qmma_max_m, qmma_tiles_per_warp, stall_test_us, qmma_operands)
    _check(lib().w4a8_set_tuning(ctypes.byref(t)))


PLAN_FIELDS = ("splits", "threads_per_row", "cols_per_thread", "rows_per_stage", "ctas_per_split",
               "grid", "rows_per_cta", "stages", "stage_bytes", "smem_bytes", "ws_bytes",
               "kernel")


def w4a8_plan_info(M: int, K: int, N: int, w8a16: bool = False, num_sms: int = 0) -> dict:
    """Launch plan for a shape; num_sms > 0 plans without a GPU."""
    arr = (ctypes.c_int * len(PLAN_FIELDS))()
    _check(lib().w4a8_plan_info(M, K, N, int(w8a16), num_sms, arr, len(PLAN_FIELDS)))
    return dict(zip(PLAN_FIELDS, list(arr)))


# group scales: the fold chunks of the fixed-order contract (count, codes each)
GROUP_PLAN_FIELDS = PLAN_FIELDS + ("chunks", "chunk_codes")


def w4a8g_plan_info(M: int, K: int, N: int, group: int, num_sms: int = 0) -> dict:
    """Launch plan of the group-scale entry points; num_sms > 0 plans without a GPU."""
    arr = (ctypes.c_int * len(GROUP_PLAN_FIELDS))()
    _check(lib().w4a8g_plan_info(M, K, N, group, num_sms, arr, len(GROUP_PLAN_FIELDS)))
    return dict(zip(GROUP_PLAN_FIELDS, list(arr)))
