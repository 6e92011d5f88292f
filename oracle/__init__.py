"""CPU oracle for the shape-driven fp16 GEMM and the M=1 decode GEMV.

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
benchmark's CPU-baseline leg may import this package; the product path
(``shape_driven_tile_gb300``) never does, and the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, fp64 accumulation); this module
compiles it with gcc on first use and wraps it with ctypes over numpy arrays of
raw bit patterns (uint16 for fp16/bf16, int8 for q8 weights).

Every entry cites the passage it follows in ``oracle.c``.  Summary:

* ``gemm(A, B, rows=None)`` -- C = A.B exactly as the definition reads
  ("Beating hipBLASLt on a Gaming GPU", section "The result").
* ``gemv_bf16(x, W)``, ``gemv_q8(x, q, s)`` -- the M=1 decode products of
  "mojo-baro", section "Four rounds on the decode shape" (rounds v1/v2).
* ``f16_to_f64``, ``bf16_to_f64``, ``f64_to_f16``, ``f64_to_bf16`` -- format conversions from
  the IEEE 754 binary16 / bfloat16 definitions.
* ``tiles`` submodule -- the tile-feasibility rules and the block-count tile
  rule of the pages, as plain integer functions.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c99", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it (gcc, no GPU)."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _bind(lib):
    i64, p = ctypes.c_int64, ctypes.c_void_p
    lib.sdt_oracle_gemm_rows.argtypes = [i64, i64, i64, p, p, p, i64, p, ctypes.c_int]
    lib.sdt_oracle_gemm_rows.restype = ctypes.c_int
    lib.sdt_oracle_gemm_rows_t.argtypes = [i64, i64, i64, p, p, p, i64, p, ctypes.c_int, ctypes.c_int]
    lib.sdt_oracle_gemm_rows_t.restype = ctypes.c_int
    lib.sdt_oracle_f64_array_to_bf16.argtypes = [p, p, i64]
    lib.sdt_oracle_gemv_bf16.argtypes = [i64, i64, p, p, p, ctypes.c_int]
    lib.sdt_oracle_gemv_bf16.restype = ctypes.c_int
    lib.sdt_oracle_gemv_q8.argtypes = [i64, i64, p, p, p, p, ctypes.c_int]
    lib.sdt_oracle_gemv_q8.restype = ctypes.c_int
    lib.sdt_oracle_f16_array_to_f64.argtypes = [p, p, i64]
    lib.sdt_oracle_bf16_array_to_f64.argtypes = [p, p, i64]
    lib.sdt_oracle_f64_array_to_f16.argtypes = [p, p, i64]
    lib.sdt_oracle_max_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _use_library(path):
    """Swap the loaded oracle for another build of it (used by the mutation tests)."""
    global _lib
    with _lock:
        prev = _lib
        _lib = _bind(ctypes.CDLL(path))
    return prev


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected uint16 bit patterns, got {a.dtype}")
    return a


def max_threads() -> int:
    return int(_load().sdt_oracle_max_threads())


def gemm(A, B, rows=None, threads: int = 0, dtype: str = "f16") -> np.ndarray:
    """fp64 C (or the selected rows of C) for 16-bit patterns A [M,K], B [K,N] (dtype f16 or bf16)."""
    A, B = _u16(A), _u16(B)
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    if rows is None:
        r = None
        n_rows = M
    else:
        r = np.ascontiguousarray(rows, dtype=np.int64)
        n_rows = r.size
    C = np.empty((n_rows, N), dtype=np.float64)
    if dtype not in ("f16", "bf16"):
        raise ValueError("dtype must be f16 or bf16")
    rc = _load().sdt_oracle_gemm_rows_t(M, N, K, _ptr(A), _ptr(B),
                                        None if r is None else _ptr(r), n_rows,
                                        _ptr(C), threads, 1 if dtype == "bf16" else 0)
    if rc != 0:
        raise ValueError("oracle gemm rejected its arguments")
    return C


def gemv_bf16(x, W, threads: int = 0) -> np.ndarray:
    """fp64 y[N] = W[N,K] . x[K] for bf16 bit patterns (W stored K-major)."""
    x, W = _u16(x), _u16(W)
    N, K = W.shape
    if x.shape != (K,):
        raise ValueError("x must have length K")
    y = np.empty(N, dtype=np.float64)
    if _load().sdt_oracle_gemv_bf16(K, N, _ptr(x), _ptr(W), _ptr(y), threads) != 0:
        raise ValueError("oracle gemv_bf16 rejected its arguments")
    return y


def gemv_q8(x, q, s, threads: int = 0) -> np.ndarray:
    """fp64 y[n] = sum_g s[n,g] * sum_{k in g} x[k] q[n,k] (groups of 32 along K)."""
    x, s = _u16(x), _u16(s)
    q = np.ascontiguousarray(q)
    if q.dtype != np.int8:
        raise TypeError("q must be int8")
    N, K = q.shape
    if x.shape != (K,) or s.shape != (N, K // 32) or K % 32:
        raise ValueError("shape mismatch (x [K], q [N,K], s [N,K/32], K % 32 == 0)")
    y = np.empty(N, dtype=np.float64)
    if _load().sdt_oracle_gemv_q8(K, N, _ptr(x), _ptr(q), _ptr(s), _ptr(y), threads) != 0:
        raise ValueError("oracle gemv_q8 rejected its arguments")
    return y


def f16_to_f64(h) -> np.ndarray:
    h = _u16(h)
    out = np.empty(h.shape, dtype=np.float64)
    _load().sdt_oracle_f16_array_to_f64(_ptr(h), _ptr(out), h.size)
    return out


def bf16_to_f64(h) -> np.ndarray:
    h = _u16(h)
    out = np.empty(h.shape, dtype=np.float64)
    _load().sdt_oracle_bf16_array_to_f64(_ptr(h), _ptr(out), h.size)
    return out


def f64_to_bf16(x) -> np.ndarray:
    """Round fp64 values to bfloat16 bit patterns, nearest, ties to even."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().sdt_oracle_f64_array_to_bf16(_ptr(x), _ptr(out), x.size)
    return out


def f64_to_f16(x) -> np.ndarray:
    """Round fp64 values to binary16 bit patterns, nearest, ties to even."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().sdt_oracle_f64_array_to_f16(_ptr(x), _ptr(out), x.size)
    return out
