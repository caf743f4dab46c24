"""CPU oracle for the tiled matrix multiply P = M x N (test infrastructure).

This package is test infrastructure.  Only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it.  The
product path (``libtgemm`` and ``dense_tiled_matrix_gb300``) never imports,
links or calls anything in here, and nothing in here imports the product.

Contents
--------
``oracle.c``  -- the fp64 triple loop (hecess.blogspot.com "[Multi-Core & GPU
                 Programming] CUDA - Matrix Multiplication", section
                 "[Matrix Multiplication]"), compiled with the host C compiler
                 into ``liboracle.so`` and called through ctypes here.
``tiled.py``  -- a pure-Python walk through the pages' shared-memory tiled
                 algorithm (same page, section "[Shared Memory]", work flow of
                 Block(0,0) and "Memory 분석"), used to pin the oracle and the
                 load-count model on small cases.

The products return fp64 results: P(i,j) = sum_k M(i,k) N(k,j) and the error
scale D(i,j) = sum_k |M(i,k)| |N(k,j)|.  ``transpose`` is the plain definition
T(j,i) = M(i,j) of the lecture's transpose case study (note.jhbae.stream
"Lec 29 · GPU Architecture (2)"), used to check the transpose kernels.
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
_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off"]

_lock = threading.Lock()
_lib = None

F64, F32, BF16 = 0, 1, 2


def compile_library(src: str = _SRC, out: str = _LIB, extra_flags=()) -> str:
    """Compile ``src`` with the host C compiler into the shared library ``out``."""
    cc = os.environ.get("CC", "cc")
    cmd = [cc, *_CFLAGS, *extra_flags, src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def build(force: bool = False) -> str:
    """Build ``liboracle.so`` next to its source if missing or stale."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        compile_library()
    return _LIB


def _bind(lib):
    i64, vp, dp = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
    lib.oracle_gemm.argtypes = [i64, i64, i64, vp, i64, ctypes.c_int, vp, i64, ctypes.c_int,
                                dp, dp, i64, ctypes.c_int]
    lib.oracle_gemm.restype = ctypes.c_int
    lib.oracle_gemm_entries.argtypes = [i64, i64, i64, vp, i64, ctypes.c_int, vp, i64,
                                        ctypes.c_int, vp, vp, i64, dp, dp]
    lib.oracle_gemm_entries.restype = ctypes.c_int
    lib.oracle_available_cores.argtypes = []
    lib.oracle_available_cores.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library; ``path`` loads another build."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def _code(a: np.ndarray) -> int:
    if a.dtype == np.float64:
        return F64
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:   # bf16 bit patterns
        return BF16
    raise TypeError(f"oracle: unsupported input dtype {a.dtype}")


def _rowmajor(a: np.ndarray) -> np.ndarray:
    """A 2-D view with unit column stride and a whole-element row stride (copies otherwise)."""
    if a.ndim != 2:
        raise ValueError("oracle: inputs must be 2-D")
    if a.strides[1] != a.itemsize or a.strides[0] % a.itemsize or a.strides[0] < 0:
        a = np.ascontiguousarray(a)
    return a


def _ld(a: np.ndarray) -> int:
    return a.strides[0] // a.itemsize if a.shape[0] > 1 else max(a.shape[1], 1)


def available_cores(lib=None) -> int:
    """Host cores this process may use (sched_getaffinity)."""
    return int((lib or load()).oracle_available_cores())


def gemm(M: np.ndarray, N: np.ndarray, nthreads: int = 0, lib=None):
    """Full product in fp64: returns ``(P, D)``, both ``m x n`` float64 arrays.

    ``M`` is ``m x k`` and ``N`` is ``k x n``; each may be float64, float32, or
    uint16 holding bf16 bit patterns.  Row-major views with any leading
    dimension are accepted.
    """
    lib = lib or load()
    M, N = _rowmajor(M), _rowmajor(N)
    m, k = M.shape
    k2, n = N.shape
    if k != k2:
        raise ValueError(f"oracle: inner dimensions differ ({k} vs {k2})")
    P = np.empty((m, n), dtype=np.float64)
    D = np.empty((m, n), dtype=np.float64)
    if m == 0 or n == 0:
        return P, D
    ldm = _ld(M) if k > 0 else max(k, 1)
    ldn = _ld(N) if k > 0 else max(n, 1)
    rc = lib.oracle_gemm(m, n, k, M.ctypes.data if k else None, ldm, _code(M),
                         N.ctypes.data if k else None, ldn, _code(N),
                         P.ctypes.data, D.ctypes.data, n, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm failed with code {rc}")
    return P, D


def gemm_entries(M: np.ndarray, N: np.ndarray, rows, cols, lib=None):
    """Chosen entries only: returns ``(P, D)`` for each pair ``(rows[c], cols[c])``."""
    lib = lib or load()
    M, N = _rowmajor(M), _rowmajor(N)
    m, k = M.shape
    k2, n = N.shape
    if k != k2:
        raise ValueError(f"oracle: inner dimensions differ ({k} vs {k2})")
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape:
        raise ValueError("oracle: rows and cols differ in length")
    P = np.empty(rows.size, dtype=np.float64)
    D = np.empty(rows.size, dtype=np.float64)
    if rows.size == 0:
        return P, D
    ldm = _ld(M) if k > 0 else max(k, 1)
    ldn = _ld(N) if k > 0 else max(n, 1)
    rc = lib.oracle_gemm_entries(m, n, k, M.ctypes.data if k else None, ldm, _code(M),
                                 N.ctypes.data if k else None, ldn, _code(N),
                                 rows.ctypes.data, cols.ctypes.data, rows.size,
                                 P.ctypes.data, D.ctypes.data)
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_entries failed with code {rc}")
    return P, D


def transpose(M: np.ndarray) -> np.ndarray:
    """T with T[j, i] = M[i, j] (numpy's transpose, materialised), same dtype."""
    M = np.asarray(M)
    if M.ndim != 2:
        raise ValueError("oracle: transpose takes a 2-D array")
    return np.ascontiguousarray(M.T)
