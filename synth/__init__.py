"""Seeded synthetic inputs shared by the oracle tests and the GPU path.

This module holds none of the method's arithmetic: it only draws numbers.
Both sides of every parity test take their inputs from here, so the CPU
oracle and the CUDA library see bit-identical data.

Generator (counter-based, so any element can be drawn on its own):

* ``fmix32`` is the 32-bit avalanche finaliser of MurmurHash3.
* ``word(seed, i, j) = fmix32(fmix32(i ^ fmix32(seed)) + (j+1)*0x9E3779B9)``
  (all arithmetic mod 2**32) is draw ``j`` of element ``i`` of stream ``seed``.
* A standard normal deviate is approximated by the Irwin-Hall sum of twelve
  uniforms: the twelve 16-bit halves ``u`` of draws ``j = 0..5`` give
  ``z = (sum(u) - 393210) / 65536``, i.e. ``sum((u + 0.5)/65536) - 6``.  It has
  mean 0 and variance ``1 - 2**-32`` and is exactly representable in binary32,
  so CPU and GPU produce the same bits.  Tails are cut at +-6 sigma.
* ``N(0, sigma)`` samples are ``float32(z) * float32(sigma)`` (one IEEE
  multiply).

``synth_gen.cu`` implements the same generator as a CUDA kernel for the large
weight tensors (random access, identical bits); ``tests/test_synth.py`` and the
GPU tests check the two agree.
"""
from __future__ import annotations

import numpy as np

GOLDEN = np.uint32(0x9E3779B9)
IH_OFFSET = 393210  # 6 * 65536 - 6: centres the sum of twelve (u + 0.5)/65536
OUTLIER_DRAW = 6    # draw index used to rank outlier positions


def fmix32(h: np.ndarray) -> np.ndarray:
    h = np.asarray(h, dtype=np.uint32).copy()
    h ^= h >> np.uint32(16)
    h *= np.uint32(0x85EBCA6B)
    h ^= h >> np.uint32(13)
    h *= np.uint32(0xC2B2AE35)
    h ^= h >> np.uint32(16)
    return h


def seed_key(seed: int) -> np.uint32:
    return fmix32(np.array([seed & 0xFFFFFFFF], np.uint32))[0]


def word(seed: int, i: np.ndarray, j: int) -> np.ndarray:
    """Draw ``j`` of elements ``i`` (uint32 counters) of stream ``seed``."""
    i = np.asarray(i)
    if i.size and (int(i.max()) >= 2**32 or int(i.min()) < 0):
        raise ValueError("counter out of the 32-bit range")
    a = fmix32(i.astype(np.uint32) ^ seed_key(seed))
    return fmix32(a + np.uint32(((j + 1) * int(GOLDEN)) & 0xFFFFFFFF))


def normal_z(seed: int, i: np.ndarray) -> np.ndarray:
    """Irwin-Hall(12) standard-normal approximation at counters ``i`` (float32)."""
    i = np.asarray(i)
    s = np.zeros(i.shape, np.int64)
    for j in range(6):
        w = word(seed, i, j)
        s += (w & np.uint32(0xFFFF)).astype(np.int64) + (w >> np.uint32(16)).astype(np.int64)
    return ((s - IH_OFFSET).astype(np.float32) / np.float32(65536.0)).astype(np.float32)


def normal(seed: int, shape, sigma: float = 1.0, offset: int = 0) -> np.ndarray:
    """Row-major tensor of N(0, sigma) samples; element e uses counter offset+e."""
    n = int(np.prod(shape))
    z = normal_z(seed, np.arange(offset, offset + n, dtype=np.int64))
    return (z * np.float32(sigma)).reshape(shape)


def weight_rows(seed: int, N: int, K: int, rows, sigma: float = 0.02) -> np.ndarray:
    """Rows ``rows`` of the [N][K] weight tensor ``normal(seed, (N, K), sigma)``."""
    rows = np.asarray(rows, dtype=np.int64)
    if rows.size and (rows.min() < 0 or rows.max() >= N):
        raise IndexError("row out of range")
    idx = rows[:, None] * K + np.arange(K, dtype=np.int64)[None, :]
    return normal_z(seed, idx) * np.float32(sigma)


def activation(seed: int, M: int, K: int, outlier_frac: float = 0.0,
               outlier_mult: float = 20.0) -> np.ndarray:
    """[M][K] binary16 activation: N(0,1), and in each row exactly
    ceil(outlier_frac*K) positions (the smallest ranking draws) scaled by
    ``outlier_mult``, then rounded to binary16 (ties to even)."""
    x = normal(seed, (M, K), 1.0)
    if outlier_frac > 0.0:
        n_out = int(np.ceil(outlier_frac * K - 1e-9))
        for m in range(M):
            keys = word(seed, np.arange(m * K, (m + 1) * K, dtype=np.int64), OUTLIER_DRAW)
            pos = np.argsort(keys, kind="stable")[:n_out]
            x[m, pos] *= np.float32(outlier_mult)
    return x.astype(np.float16)


def n_outliers(K: int, outlier_frac: float) -> int:
    return int(np.ceil(outlier_frac * K - 1e-9)) if outlier_frac > 0 else 0


# ----------------------------------------------------------------------------
# CUDA twin of ``normal`` for large tensors (test / benchmark infrastructure)
# ----------------------------------------------------------------------------

import ctypes as _ct
import os as _os
import subprocess as _sp

_HERE = _os.path.dirname(_os.path.abspath(__file__))
_CU = _os.path.join(_HERE, "synth_gen.cu")
_SO = _os.path.join(_HERE, "_build", "libsynth.so")
_LIB = None


def build_gpu() -> str:
    """Compile libsynth.so for sm_103a if it is missing or stale."""
    if _os.path.exists(_SO) and _os.path.getmtime(_SO) >= _os.path.getmtime(_CU):
        return _SO
    _os.makedirs(_os.path.dirname(_SO), exist_ok=True)
    nvcc = _os.path.join(_os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    tmp = _SO + ".tmp%d" % _os.getpid()
    _sp.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-Xcompiler", "-fPIC", "-shared", "-cudart", "static", "-o", tmp, _CU])
    _os.replace(tmp, _SO)
    return _SO


def _gpu_lib():
    global _LIB
    if _LIB is None:
        lib = _ct.CDLL(build_gpu())
        lib.synth_normal_f32.restype = _ct.c_int
        lib.synth_normal_f32.argtypes = [_ct.c_uint32, _ct.c_uint64, _ct.c_uint64, _ct.c_float,
                                         _ct.c_void_p, _ct.c_void_p]
        _LIB = lib
    return _LIB


def normal_gpu(seed: int, shape, sigma: float = 1.0, offset: int = 0, device="cuda", out=None):
    """Same values as ``normal(seed, shape, sigma, offset)``, drawn on the GPU
    into a float32 torch tensor."""
    import torch
    n = int(np.prod(shape))
    if out is None:
        out = torch.empty(tuple(shape), dtype=torch.float32, device=device)
    assert out.dtype == torch.float32 and out.is_contiguous() and out.numel() == n
    stream = torch.cuda.current_stream(out.device).cuda_stream
    st = _gpu_lib().synth_normal_f32(seed & 0xFFFFFFFF, offset, n, float(np.float32(sigma)),
                                      out.data_ptr(), stream)
    if st != 0:
        raise RuntimeError("synth_normal_f32 failed with status %d" % st)
    return out


# ----------------------------------------------------------------------------
# C twin of ``normal`` on the host, split over threads (test infrastructure)
# ----------------------------------------------------------------------------

_HOST_C = _os.path.join(_HERE, "synth_host.c")
_HOST_SO = _os.path.join(_HERE, "_build", "libsynth_host.so")
_HOST_LIB = None


def build_host() -> str:
    """Compile libsynth_host.so with gcc if it is missing or stale."""
    if _os.path.exists(_HOST_SO) and _os.path.getmtime(_HOST_SO) >= _os.path.getmtime(_HOST_C):
        return _HOST_SO
    _os.makedirs(_os.path.dirname(_HOST_SO), exist_ok=True)
    tmp = _HOST_SO + ".tmp%d" % _os.getpid()
    _sp.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    "-o", tmp, _HOST_C])
    _os.replace(tmp, _HOST_SO)
    return _HOST_SO


def _host_lib():
    global _HOST_LIB
    if _HOST_LIB is None:
        lib = _ct.CDLL(build_host())
        lib.synth_normal_f32_host.restype = _ct.c_int
        lib.synth_normal_f32_host.argtypes = [_ct.c_uint32, _ct.c_uint64, _ct.c_uint64, _ct.c_float,
                                              _ct.c_void_p, _ct.c_int]
        _HOST_LIB = lib
    return _HOST_LIB


def normal_host(seed: int, shape, sigma: float = 1.0, offset: int = 0, threads: int = 0) -> np.ndarray:
    """Same values as ``normal(seed, shape, sigma, offset)``, drawn by the C
    twin over ``threads`` host threads (0 = every core)."""
    n = int(np.prod(shape))
    out = np.empty(n, np.float32)
    th = threads if threads > 0 else (_os.cpu_count() or 1)
    st = _host_lib().synth_normal_f32_host(seed & 0xFFFFFFFF, offset, n, float(np.float32(sigma)),
                                           out.ctypes.data, th)
    if st != 0:
        raise ValueError("synth_normal_f32_host failed with status %d" % st)
    return out.reshape(shape)
