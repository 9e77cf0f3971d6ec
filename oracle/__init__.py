"""CPU oracle for the W4A8 / W8A16 decode linear -- TEST INFRASTRUCTURE ONLY.

A plain, single-threaded C definition (``oracle.c``) of what the hot path
computes, loaded with ctypes and wrapped for numpy arrays.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package; the product library never does.  It shares no code with the
CUDA library.

Every function cites the passage of the pages it follows in ``oracle.c``.
No function here is "parity unpinned": the pins live in
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")

CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

OK = 0
ERR_SHAPE = 3
ERR_OVERFLOW = 6


def compile_oracle(src: str = _SRC, out: str = _LIB, extra=()) -> str:
    """Compile ``src`` into the shared library ``out`` with gcc (no FMA
    contraction); ``extra`` adds flags (e.g. sanitizers)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", *CFLAGS, *extra, "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def build() -> str:
    """Build ``liboracle.so`` if it is missing or older than ``oracle.c``."""
    if not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        compile_oracle()
    return _LIB


_i64 = ctypes.c_int64
_p = ctypes.c_void_p


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        self._lib = lib
        lib.oracle_half_to_float.restype = ctypes.c_float
        lib.oracle_half_to_float.argtypes = [ctypes.c_uint16]
        lib.oracle_float_to_half.restype = ctypes.c_uint16
        lib.oracle_float_to_half.argtypes = [ctypes.c_float]
        for name, args in {
            "oracle_w4_quantize": [_p, _i64, _i64, _p, _p],
            "oracle_w4_unpack": [_p, _i64, _i64, _p],
            "oracle_act_quantize": [_p, _i64, _i64, _p, _p],
            "oracle_w4a8_dot": [_p, _i64, _i64, _p, _i64, _p],
            "oracle_w4a8_linear": [_p, _i64, _i64, _p, _p, _i64, _p, _p, _p, _p],
            "oracle_w8_quantize": [_p, _i64, _i64, _p, _p],
            "oracle_w4g_quantize": [_p, _i64, _i64, _i64, _p, _p],
            "oracle_w4a8g_ref": [_p, _p, _i64, _i64, _i64, _p, _p, _i64, _p, _p],
            "oracle_w4a8g_linear": [_p, _i64, _i64, _i64, _p, _p, _i64, _p, _p, _p, _p],
            "oracle_w4a8g_f32": [_p, _p, _i64, _i64, _i64, _p, _p, _i64, _p],
            "oracle_w4a8g_linear_f32": [_p, _i64, _i64, _i64, _p, _p, _i64, _p, _p, _p],
            "oracle_isx_lut": [ctypes.c_int, ctypes.c_double, _p],
            "oracle_index_softmax": [_p, _i64, _i64, _i64, ctypes.c_int, _p, _p],
        }.items():
            f = getattr(lib, name)
            f.restype = ctypes.c_int
            f.argtypes = args
        lib.oracle_w4a8_rescale.restype = None
        lib.oracle_w4a8_rescale.argtypes = [_p, _p, _p, _i64, _i64, _p]
        lib.oracle_w4g_scale_stride.restype = _i64
        lib.oracle_w4g_scale_stride.argtypes = [_i64, _i64]
        lib.oracle_isx_c_int.restype = _i64
        lib.oracle_isx_c_int.argtypes = [ctypes.c_double, _i64, ctypes.c_float, ctypes.c_float]
        lib.oracle_w8a16_ref.restype = None
        lib.oracle_w8a16_ref.argtypes = [_p, _i64, _i64, _p, _p, _i64, _p]
        lib.oracle_double_to_half.restype = ctypes.c_uint16
        lib.oracle_double_to_half.argtypes = [ctypes.c_double]
        lib.oracle_silu_mul.restype = None
        lib.oracle_silu_mul.argtypes = [_p, _p, _i64, _p, _p]

    # -- binary16 ---------------------------------------------------------
    def half_to_float(self, bits: int) -> float:
        return self._lib.oracle_half_to_float(int(bits))

    def float_to_half(self, x: float) -> int:
        return int(self._lib.oracle_float_to_half(float(np.float32(x))))

    def double_to_half(self, x: float) -> int:
        return int(self._lib.oracle_double_to_half(float(x)))

    # -- the MLP's gated product ---------------------------------------------
    def silu_mul(self, g: np.ndarray, u: np.ndarray):
        """(v, h): v = silu(g) * u in binary64, h its binary16 bits (uint16)."""
        g = np.ascontiguousarray(g, dtype=np.float32)
        u = np.ascontiguousarray(u, dtype=np.float32)
        assert g.shape == u.shape
        v = np.empty(g.shape, np.float64)
        h = np.empty(g.shape, np.uint16)
        self._lib.oracle_silu_mul(_ptr(g), _ptr(u), g.size, _ptr(v), _ptr(h))
        return v, h

    # -- W4A8 -------------------------------------------------------------
    def w4_quantize(self, W: np.ndarray):
        W = np.ascontiguousarray(W, dtype=np.float32)
        N, K = W.shape
        Wq = np.empty((N, K // 2), np.uint8)
        sw = np.empty(N, np.float32)
        st = self._lib.oracle_w4_quantize(_ptr(W), N, K, _ptr(Wq), _ptr(sw))
        if st != OK:
            raise ValueError("oracle_w4_quantize status %d" % st)
        return Wq, sw

    def w4_unpack(self, Wq: np.ndarray, K: int) -> np.ndarray:
        Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
        N = Wq.shape[0]
        q = np.empty((N, K), np.int8)
        st = self._lib.oracle_w4_unpack(_ptr(Wq), N, K, _ptr(q))
        if st != OK:
            raise ValueError("oracle_w4_unpack status %d" % st)
        return q

    def act_quantize(self, X: np.ndarray):
        X = np.ascontiguousarray(X, dtype=np.float16)
        M, K = X.shape
        Xq = np.empty((M, K), np.int8)
        sa = np.empty(M, np.float32)
        st = self._lib.oracle_act_quantize(_ptr(X), M, K, _ptr(Xq), _ptr(sa))
        if st != OK:
            raise ValueError("oracle_act_quantize status %d" % st)
        return Xq, sa

    def w4a8_dot(self, Xq: np.ndarray, Wq: np.ndarray) -> np.ndarray:
        Xq = np.ascontiguousarray(Xq, dtype=np.int8)
        Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
        M, K = Xq.shape
        N = Wq.shape[0]
        assert Wq.shape[1] * 2 == K
        acc = np.empty((M, N), np.int32)
        st = self._lib.oracle_w4a8_dot(_ptr(Xq), M, K, _ptr(Wq), N, _ptr(acc))
        if st != OK:
            raise OverflowError("oracle_w4a8_dot status %d" % st)
        return acc

    def w4a8_rescale(self, acc: np.ndarray, sw: np.ndarray, sa: np.ndarray) -> np.ndarray:
        acc = np.ascontiguousarray(acc, dtype=np.int32)
        sw = np.ascontiguousarray(sw, dtype=np.float32)
        sa = np.ascontiguousarray(sa, dtype=np.float32)
        M, N = acc.shape
        Y = np.empty((M, N), np.float32)
        self._lib.oracle_w4a8_rescale(_ptr(acc), _ptr(sw), _ptr(sa), M, N, _ptr(Y))
        return Y

    def w4a8_linear(self, X: np.ndarray, Wq: np.ndarray, sw: np.ndarray):
        """Returns (Y, Xq, sa, acc)."""
        X = np.ascontiguousarray(X, dtype=np.float16)
        Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
        sw = np.ascontiguousarray(sw, dtype=np.float32)
        M, K = X.shape
        N = Wq.shape[0]
        assert Wq.shape[1] * 2 == K
        Y = np.empty((M, N), np.float32)
        Xq = np.empty((M, K), np.int8)
        sa = np.empty(M, np.float32)
        acc = np.empty((M, N), np.int32)
        st = self._lib.oracle_w4a8_linear(_ptr(X), M, K, _ptr(Wq), _ptr(sw), N, _ptr(Y),
                                          _ptr(Xq), _ptr(sa), _ptr(acc))
        if st != OK:
            raise OverflowError("oracle_w4a8_linear status %d" % st)
        return Y, Xq, sa, acc

    # -- group-wise W4A8 --------------------------------------------------
    def w4g_scale_stride(self, K: int, gs: int) -> int:
        return int(self._lib.oracle_w4g_scale_stride(K, gs))

    def w4g_quantize(self, W: np.ndarray, gs: int):
        """Returns (Wq [N][K/2] uint8, sg [N][stride] float32)."""
        W = np.ascontiguousarray(W, dtype=np.float32)
        N, K = W.shape
        Wq = np.empty((N, K // 2), np.uint8)
        sg = np.empty((N, max(1, self.w4g_scale_stride(K, gs))), np.float32)
        st = self._lib.oracle_w4g_quantize(_ptr(W), N, K, gs, _ptr(Wq), _ptr(sg))
        if st != OK:
            raise ValueError("oracle_w4g_quantize status %d" % st)
        return Wq, sg

    def w4a8g_ref(self, Xq: np.ndarray, sa: np.ndarray, Wq: np.ndarray, sg: np.ndarray, gs: int):
        """Returns (Y, B) in float64: the product and its rounding magnitude."""
        Xq = np.ascontiguousarray(Xq, dtype=np.int8)
        sa = np.ascontiguousarray(sa, dtype=np.float32)
        Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
        sg = np.ascontiguousarray(sg, dtype=np.float32)
        M, K = Xq.shape
        N = Wq.shape[0]
        assert Wq.shape[1] * 2 == K and sg.shape == (N, self.w4g_scale_stride(K, gs))
        Y = np.empty((M, N), np.float64)
        B = np.empty((M, N), np.float64)
        st = self._lib.oracle_w4a8g_ref(_ptr(Xq), _ptr(sa), M, K, gs, _ptr(Wq), _ptr(sg), N,
                                        _ptr(Y), _ptr(B))
        if st != OK:
            raise ValueError("oracle_w4a8g_ref status %d" % st)
        return Y, B

    def w4a8g_linear(self, X: np.ndarray, Wq: np.ndarray, sg: np.ndarray, gs: int):
        """Returns (Y, B, Xq, sa)."""
        X = np.ascontiguousarray(X, dtype=np.float16)
        Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
        sg = np.ascontiguousarray(sg, dtype=np.float32)
        M, K = X.shape
        N = Wq.shape[0]
        assert Wq.shape[1] * 2 == K and sg.shape == (N, self.w4g_scale_stride(K, gs))
        Y = np.empty((M, N), np.float64)
        B = np.empty((M, N), np.float64)
        Xq = np.empty((M, K), np.int8)
        sa = np.empty(M, np.float32)
        st = self._lib.oracle_w4a8g_linear(_ptr(X), M, K, gs, _ptr(Wq), _ptr(sg), N, _ptr(Y),
                                           _ptr(B), _ptr(Xq), _ptr(sa))
        if st != OK:
            raise ValueError("oracle_w4a8g_linear status %d" % st)
        return Y, B, Xq, sa

    def w4a8g_f32(self, Xq: np.ndarray, sa: np.ndarray, Wq: np.ndarray, sg: np.ndarray, gs: int):
        """The group-wise product in the fixed binary32 order: Y [M][N] fp32."""
        Xq = np.ascontiguousarray(Xq, dtype=np.int8)
        sa = np.ascontiguousarray(sa, dtype=np.float32)
        Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
        sg = np.ascontiguousarray(sg, dtype=np.float32)
        M, K = Xq.shape
        N = Wq.shape[0]
        assert Wq.shape[1] * 2 == K and sg.shape == (N, self.w4g_scale_stride(K, gs))
        Y = np.empty((M, N), np.float32)
        st = self._lib.oracle_w4a8g_f32(_ptr(Xq), _ptr(sa), M, K, gs, _ptr(Wq), _ptr(sg), N, _ptr(Y))
        if st != OK:
            raise ValueError("oracle_w4a8g_f32 status %d" % st)
        return Y

    def w4a8g_linear_f32(self, X: np.ndarray, Wq: np.ndarray, sg: np.ndarray, gs: int):
        """Returns (Y fp32 in the fixed order, Xq, sa)."""
        X = np.ascontiguousarray(X, dtype=np.float16)
        Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
        sg = np.ascontiguousarray(sg, dtype=np.float32)
        M, K = X.shape
        N = Wq.shape[0]
        assert Wq.shape[1] * 2 == K and sg.shape == (N, self.w4g_scale_stride(K, gs))
        Y = np.empty((M, N), np.float32)
        Xq = np.empty((M, K), np.int8)
        sa = np.empty(M, np.float32)
        st = self._lib.oracle_w4a8g_linear_f32(_ptr(X), M, K, gs, _ptr(Wq), _ptr(sg), N, _ptr(Y),
                                               _ptr(Xq), _ptr(sa))
        if st != OK:
            raise ValueError("oracle_w4a8g_linear_f32 status %d" % st)
        return Y, Xq, sa

    # -- IndexSoftmax -----------------------------------------------------
    def isx_lut(self, b: int = 5, c: float = 6.6) -> np.ndarray:
        lut = np.empty(1 << b, np.uint8)
        st = self._lib.oracle_isx_lut(b, c, _ptr(lut))
        if st != OK:
            raise ValueError("oracle_isx_lut status %d" % st)
        return lut

    def isx_c_int(self, c: float, d: int, s_q: float, s_k: float) -> int:
        return int(self._lib.oracle_isx_c_int(c, d, float(np.float32(s_q)), float(np.float32(s_k))))

    def index_softmax(self, A: np.ndarray, c_int: int, b: int = 5, lut=None) -> np.ndarray:
        """int32 logits [rows][cols] -> UINT8 probabilities (same shape)."""
        A = np.ascontiguousarray(A, dtype=np.int32)
        rows, cols = A.shape
        lut = self.isx_lut(b) if lut is None else np.ascontiguousarray(lut, dtype=np.uint8)
        P = np.empty((rows, cols), np.uint8)
        st = self._lib.oracle_index_softmax(_ptr(A), rows, cols, c_int, b, _ptr(lut), _ptr(P))
        if st != OK:
            raise ValueError("oracle_index_softmax status %d" % st)
        return P

    # -- W8A16 ------------------------------------------------------------
    def w8_quantize(self, W: np.ndarray):
        W = np.ascontiguousarray(W, dtype=np.float32)
        N, K = W.shape
        Wq8 = np.empty((N, K), np.int8)
        sw16 = np.empty(N, np.float16)
        st = self._lib.oracle_w8_quantize(_ptr(W), N, K, _ptr(Wq8), _ptr(sw16))
        if st != OK:
            raise ValueError("oracle_w8_quantize status %d" % st)
        return Wq8, sw16

    def w8a16_ref(self, X: np.ndarray, Wq8: np.ndarray, sw16: np.ndarray) -> np.ndarray:
        X = np.ascontiguousarray(X, dtype=np.float16)
        Wq8 = np.ascontiguousarray(Wq8, dtype=np.int8)
        sw16 = np.ascontiguousarray(sw16, dtype=np.float16)
        M, K = X.shape
        N = Wq8.shape[0]
        assert Wq8.shape[1] == K
        Y = np.empty((M, N), np.float64)
        self._lib.oracle_w8a16_ref(_ptr(X), M, K, _ptr(Wq8), _ptr(sw16), N, _ptr(Y))
        return Y


_DEFAULT = None


def load() -> Oracle:
    """The oracle built from ``oracle.c`` (compiled on first use)."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle(build())
    return _DEFAULT
