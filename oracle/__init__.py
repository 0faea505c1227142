"""CPU oracle for the W4A16 hot path (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline / reference arm may import this package.  It loads
``liboracle.so``, built from ``w4a16_oracle.c`` by :func:`build`, and wraps
its plain binary64 loops for numpy arrays.  It shares no code with the CUDA
library and never imports it.

Weights are affine (w = scale*q + bias) or, with ``biases=None``, symmetric
(w = scale*(q - 8)); ``group`` is the quantisation group along K.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(exhaustive binary16 decode, correctly rounded encode against numpy and
Fraction arithmetic, exact-rational brute force, closed forms, invariants).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a16_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.RLock()


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (IEEE-strict: no FP contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.orc_half_to_double.restype = ctypes.c_double
            lib.orc_half_to_double.argtypes = [ctypes.c_uint16]
            lib.orc_double_to_half.restype = ctypes.c_uint16
            lib.orc_double_to_half.argtypes = [ctypes.c_double]
            lib.orc_unpack.argtypes = [P, I, I, P]
            lib.orc_dequant_exact_rows.argtypes = [P, P, P, I, I, P, I, P]
            lib.orc_dequant_f16_t.argtypes = [P, P, P, I, I, I, P]
            lib.orc_dequant_f16_rows.argtypes = [P, P, P, I, I, P, I, P]
            lib.orc_gemv_rows.argtypes = [P, P, P, P, I, I, I, P, I, P, P]
            lib.orc_topk.argtypes = [P, I, I, P, P]
            lib.orc_gemm_entries.argtypes = [P, P, I, I, P, P, I, P, P]
            lib.orc_gemm.argtypes = [P, P, I, I, I, P, P]
            for f in ("orc_unpack", "orc_dequant_exact_rows", "orc_dequant_f16_t",
                      "orc_dequant_f16_rows", "orc_gemv_rows", "orc_topk",
                      "orc_gemm_entries", "orc_gemm"):
                getattr(lib, f).restype = None
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits16(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    assert a.dtype == np.uint16
    return np.ascontiguousarray(a)


def _pb(biases):
    """Pointer to the biases, or NULL for symmetric codes (biases None)."""
    return None if biases is None else _p(_bits16(biases))


def _u32(a) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(a))
    assert a.dtype == np.uint32
    return a


def half_to_double(h: int) -> float:
    return _load().orc_half_to_double(int(h))


def double_to_half(v: float) -> int:
    return int(_load().orc_double_to_half(float(v)))


def double_to_half_array(v) -> np.ndarray:
    lib = _load()
    v = np.asarray(v, dtype=np.float64).ravel()
    return np.array([lib.orc_double_to_half(float(t)) for t in v], dtype=np.uint16)


def unpack(qweight, N: int, K: int) -> np.ndarray:
    qw = _u32(qweight)
    q = np.empty((N, K), dtype=np.uint8)
    _load().orc_unpack(_p(qw), N, K, _p(q))
    return q


def dequant_exact_rows(qweight, scales, biases, K: int, rows, group: int = 64) -> np.ndarray:
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    w = np.empty((len(rows), K), dtype=np.float64)
    _load().orc_dequant_exact_rows(_p(_u32(qweight)), _p(_bits16(scales)), _pb(biases),
                                   K, group, _p(rows), len(rows), _p(w))
    return w


def dequant_f16_t(qweight, scales, biases, N: int, K: int, group: int = 64) -> np.ndarray:
    """Transposed binary16 scratch as uint16 bits, shape [K][N]."""
    w16 = np.empty((K, N), dtype=np.uint16)
    _load().orc_dequant_f16_t(_p(_u32(qweight)), _p(_bits16(scales)), _pb(biases),
                              N, K, group, _p(w16))
    return w16


def dequant_f16_rows(qweight, scales, biases, K: int, rows, group: int = 64) -> np.ndarray:
    """Rows ``rows`` of the dequantised weight as binary16 bits, shape [len(rows)][K]."""
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    out = np.empty((len(rows), K), dtype=np.uint16)
    _load().orc_dequant_f16_rows(_p(_u32(qweight)), _p(_bits16(scales)), _pb(biases),
                                 K, group, _p(rows), len(rows), _p(out))
    return out


def gemv_rows(x, qweight, scales, biases, K: int, rows, group: int = 64):
    """(y, absdot), each [M][len(rows)] binary64, for the listed output rows."""
    x = _bits16(x).reshape(-1, K)
    M = x.shape[0]
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    y = np.empty((M, len(rows)), dtype=np.float64)
    ad = np.empty((M, len(rows)), dtype=np.float64)
    _load().orc_gemv_rows(_p(x), _p(_u32(qweight)), _p(_bits16(scales)), _pb(biases),
                          M, K, group, _p(rows), len(rows), _p(y), _p(ad))
    return y, ad


def gemv(x, qweight, scales, biases, N: int, K: int, group: int = 64, threads: int = 1):
    """Full GEMV (y, absdot), each [M][N]; ``threads`` > 1 splits rows over threads."""
    if threads <= 1:
        return gemv_rows(x, qweight, scales, biases, K, np.arange(N), group)
    from concurrent.futures import ThreadPoolExecutor
    chunks = np.array_split(np.arange(N, dtype=np.int32), threads)
    with ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(lambda r: gemv_rows(x, qweight, scales, biases, K, r, group), chunks))
    return (np.concatenate([p[0] for p in parts], axis=1),
            np.concatenate([p[1] for p in parts], axis=1))


def topk(logits, k: int):
    """(idx int32 [k], val float64 [k]) ordered by value desc, ties to lowest index."""
    lg = np.ascontiguousarray(np.asarray(logits, dtype=np.float64))
    idx = np.empty(k, dtype=np.int32)
    val = np.empty(k, dtype=np.float64)
    with _lock:
        _load().orc_topk(_p(lg), lg.size, k, _p(idx), _p(val))
    return idx, val


def gemm_entries(x16, w16, N: int, K: int, ms, ns):
    """(y, absdot) for the entries (ms[i], ns[i]) of x16[M][K] @ w16[K][N]."""
    x16 = _bits16(x16)
    w16 = _bits16(w16)
    ms = np.ascontiguousarray(np.asarray(ms, dtype=np.int32))
    ns = np.ascontiguousarray(np.asarray(ns, dtype=np.int32))
    y = np.empty(len(ms), dtype=np.float64)
    ad = np.empty(len(ms), dtype=np.float64)
    _load().orc_gemm_entries(_p(x16), _p(w16), N, K, _p(ms), _p(ns), len(ms), _p(y), _p(ad))
    return y, ad


def gemm(x16, w16, M: int, N: int, K: int):
    """(y, absdot), each [M][N] binary64, for x16[M][K] @ w16[K][N]."""
    y = np.empty((M, N), dtype=np.float64)
    ad = np.empty((M, N), dtype=np.float64)
    _load().orc_gemm(_p(_bits16(x16)), _p(_bits16(w16)), M, N, K, _p(y), _p(ad))
    return y, ad
