"""Python binding of libtgemm_pages: the pages' naive and shared-memory tiled
kernels (comparators; ``include/tgemm_pages.h``).  Argument marshalling only."""
from __future__ import annotations

import ctypes
import os
import threading

from . import tgemm as _t

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtgemm_pages.so")

_I64, _VP = ctypes.c_int64, ctypes.c_void_p
SIGNATURES = {
    "tgemm_pages_naive_f32": (ctypes.c_int, [_I64, _I64, _I64, _VP, _I64, _VP, _I64, _VP, _I64, _VP]),
    "tgemm_pages_tiled_f32": (ctypes.c_int, [_I64, _I64, _I64, _VP, _I64, _VP, _I64, _VP, _I64, ctypes.c_int,
                                             _VP]),
    "tgemm_pages_transpose_f32": (ctypes.c_int, [_I64, _I64, _VP, _I64, _VP, _I64, ctypes.c_int, _VP]),
}

_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise ImportError(f"libtgemm_pages.so not found at {path}; run dense_tiled_matrix_gb300.build.build()")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
        return _lib


def _prep(A, B, C):
    import torch
    if A.dtype != torch.float32 or B.dtype != torch.float32:
        raise TypeError("pages kernels take float32 inputs")
    m, k = int(A.shape[0]), int(A.shape[1])
    n = int(B.shape[1])
    if C is None:
        C = torch.empty((m, n), dtype=torch.float32, device=A.device)
    return m, n, k, C


def _check(status):
    if status != 0:
        raise _t.TgemmError(status, f"pages kernel failed: {_t.tgemm_status_string(status)}")


def tgemm_pages_naive_f32(A, B, C=None, stream=None):
    m, n, k, C = _prep(A, B, C)
    _check(load().tgemm_pages_naive_f32(m, n, k, A.data_ptr() or None, _t._ld(A), B.data_ptr() or None, _t._ld(B),
                                        C.data_ptr() or None, _t._ld(C), _t._stream_handle(stream)))
    return C


def tgemm_pages_tiled_f32(A, B, C=None, tile_width=16, stream=None):
    m, n, k, C = _prep(A, B, C)
    _check(load().tgemm_pages_tiled_f32(m, n, k, A.data_ptr() or None, _t._ld(A), B.data_ptr() or None, _t._ld(B),
                                        C.data_ptr() or None, _t._ld(C), int(tile_width), _t._stream_handle(stream)))
    return C


TRANSPOSE_VARIANTS = {"naive": 0, "coalesced": 1, "padded": 2}


def tgemm_pages_transpose_f32(src, dst=None, variant="padded", stream=None):
    """The lecture's transpose kernels: variant "naive", "coalesced" (tile[32][32]) or "padded" (tile[32][33])."""
    import torch
    rows, cols = int(src.shape[0]), int(src.shape[1])
    if dst is None:
        dst = torch.empty((cols, rows), dtype=torch.float32, device=src.device)
    _check(load().tgemm_pages_transpose_f32(rows, cols, src.data_ptr() or None, _t._ld(src), dst.data_ptr() or None,
                                            _t._ld(dst), TRANSPOSE_VARIANTS[variant], _t._stream_handle(stream)))
    return dst
