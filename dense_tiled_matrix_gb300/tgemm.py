"""Python binding of libtgemm (argument marshalling only).

The functions carry the names of the C entry points in ``include/tgemm.h``.
Each takes torch CUDA tensors, checks their dtype, device and layout, derives
m, n, k and the leading dimensions, and calls the C function on the current
torch stream (or the stream given).  All arithmetic happens in the library's
CUDA kernels; there is no other code path.  If ``libtgemm.so`` has not been
built, every call raises ``ImportError`` -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libtgemm.so")
# The same library built with the device-side consistency checks (TGEMM_DEBUG).
DEBUG_LIB_PATH = os.path.join(PKG, "libtgemm_debug.so")

TGEMM_OK = 0
TGEMM_ERR_INVALID_VALUE = 1
TGEMM_ERR_MISALIGNED = 2
TGEMM_ERR_UNSUPPORTED_DEVICE = 3
TGEMM_ERR_CUDA = 4
TGEMM_ERR_TIMEOUT = 5
TGEMM_ERR_WORKSPACE = 6
TGEMM_ERR_INTERNAL = 7

# Every symbol declared in include/tgemm.h, with its ctypes signature.
_I64, _VP = ctypes.c_int64, ctypes.c_void_p
_GEMM_ARGS = [_I64, _I64, _I64, _VP, _I64, _VP, _I64, _VP, _I64, _VP]
SIGNATURES = {
    "tgemm_f32": (ctypes.c_int, _GEMM_ARGS),
    "tgemm_tf32": (ctypes.c_int, _GEMM_ARGS),
    "tgemm_bf16": (ctypes.c_int, _GEMM_ARGS),
    "tgemm_tf32_noalloc": (ctypes.c_int, _GEMM_ARGS),
    "tgemm_transpose_f32": (ctypes.c_int, [_I64, _I64, _VP, _I64, _VP, _I64, _VP]),
    "tgemm_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "tgemm_last_error": (ctypes.c_char_p, []),
    "tgemm_get_device_status": (ctypes.c_int, [_VP]),
    "tgemm_selftest_wait_timeout": (ctypes.c_int, [_I64, _VP]),
    "tgemm_selftest_debug_check": (ctypes.c_int, [_VP]),
    "tgemm_debug_build": (ctypes.c_int, []),
    "tgemm_kernel_launches": (ctypes.c_uint64, []),
    "tgemm_plan": (ctypes.c_int, [ctypes.c_int, _I64, _I64, _I64, ctypes.c_int, ctypes.c_int,
                                  ctypes.POINTER(ctypes.c_int)]),
    "tgemm_plan_f32": (ctypes.c_int, [_I64, _I64, _I64, ctypes.c_int, ctypes.POINTER(ctypes.c_int64)]),
    "tgemm_version": (ctypes.c_int, []),
}

_lock = threading.Lock()
_lib = None


class TgemmError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


def open_library(path: str):
    """A ctypes handle on a libtgemm build at ``path`` with every entry point's
    signature set; raises ImportError if the file does not exist."""
    if not os.path.exists(path):
        raise ImportError(f"{os.path.basename(path)} not found at {path}; run dense_tiled_matrix_gb300.build.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load(path: str = LIB_PATH):
    """The loaded library (ctypes.CDLL); raises ImportError if it is not built."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = open_library(path)
        return _lib


def _check(status: int):
    if status != TGEMM_OK:
        lib = load()
        raise TgemmError(status, f"{lib.tgemm_status_string(status).decode()}: {lib.tgemm_last_error().decode()}")


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ld(t) -> int:
    if t.dim() != 2:
        raise ValueError("tgemm: operands must be 2-D")
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError("tgemm: operands must be row-major (unit column stride)")
    if t.shape[0] <= 1:
        return max(int(t.shape[1]), 1)
    return int(t.stride(0))


def _call(name, A, B, C, stream, in_dtype, lib=None):
    import torch
    if A.dtype != in_dtype or B.dtype != in_dtype:
        raise TypeError(f"{name}: inputs must be {in_dtype}")
    if A.shape[1] != B.shape[0]:
        raise ValueError(f"{name}: inner dimensions differ ({A.shape[1]} vs {B.shape[0]})")
    m, k = int(A.shape[0]), int(A.shape[1])
    n = int(B.shape[1])
    if C is None:
        C = torch.empty((m, n), dtype=torch.float32, device=A.device)
    if C.dtype != torch.float32 or tuple(C.shape) != (m, n):
        raise ValueError(f"{name}: C must be a float32 tensor of shape ({m}, {n})")
    for t in (A, B, C):
        if t.numel() and not t.is_cuda:
            raise ValueError(f"{name}: tensors must live on a CUDA device")
    lib = lib or load()
    status = getattr(lib, name)(m, n, k, A.data_ptr() or None, _ld(A), B.data_ptr() or None, _ld(B),
                                C.data_ptr() or None, _ld(C), _stream_handle(stream))
    if status != TGEMM_OK:
        raise TgemmError(status, f"{lib.tgemm_status_string(status).decode()}: {lib.tgemm_last_error().decode()}")
    return C


def tgemm_f32(A, B, C=None, stream=None, lib=None):
    """C = A @ B for float32 tensors on the FMA pipes (fp32 throughout)."""
    import torch
    return _call("tgemm_f32", A, B, C, stream, torch.float32, lib)


def tgemm_tf32(A, B, C=None, stream=None, lib=None):
    """C = A @ B for float32 tensors on the tensor cores as TF32, fp32 accumulation."""
    import torch
    return _call("tgemm_tf32", A, B, C, stream, torch.float32, lib)


def tgemm_bf16(A, B, C=None, stream=None, lib=None):
    """C (float32) = A @ B for bfloat16 tensors on the tensor cores, fp32 accumulation."""
    import torch
    return _call("tgemm_bf16", A, B, C, stream, torch.bfloat16, lib)


def tgemm_tf32_noalloc(A, B, C=None, stream=None, lib=None):
    """Like ``tgemm_tf32`` but with its scratch in the library's static device
    array (no allocation by the library); the shape must fit TGEMM_NOALLOC_SCRATCH_BYTES."""
    import torch
    return _call("tgemm_tf32_noalloc", A, B, C, stream, torch.float32, lib)


NOALLOC_SCRATCH_BYTES = 32 << 20


def tgemm_transpose_f32(src, dst=None, stream=None):
    """dst = src.T for a float32 CUDA matrix (row-major views with any pitch)."""
    import torch
    if src.dtype != torch.float32 or src.dim() != 2:
        raise TypeError("tgemm_transpose_f32: src must be a 2-D float32 tensor")
    rows, cols = int(src.shape[0]), int(src.shape[1])
    if dst is None:
        dst = torch.empty((cols, rows), dtype=torch.float32, device=src.device)
    if dst.dtype != torch.float32 or tuple(dst.shape) != (cols, rows):
        raise ValueError(f"tgemm_transpose_f32: dst must be float32 of shape ({cols}, {rows})")
    _check(load().tgemm_transpose_f32(rows, cols, src.data_ptr() or None, _ld(src), dst.data_ptr() or None,
                                      _ld(dst), _stream_handle(stream)))
    return dst


def tgemm_status_string(status: int) -> str:
    return load().tgemm_status_string(int(status)).decode()


def tgemm_last_error() -> str:
    return load().tgemm_last_error().decode()


def tgemm_get_device_status(stream=None) -> int:
    """Waits for ``stream`` and returns (and clears) the device status word."""
    return int(load().tgemm_get_device_status(_stream_handle(stream)))


def tgemm_selftest_wait_timeout(limit_ns: int, stream=None) -> int:
    """Queues a kernel whose bounded wait must time out after ``limit_ns``; returns the call status."""
    return int(load().tgemm_selftest_wait_timeout(int(limit_ns), _stream_handle(stream)))


def tgemm_selftest_debug_check(stream=None) -> int:
    """Queues a kernel that records a failed device check; returns the call status."""
    return int(load().tgemm_selftest_debug_check(_stream_handle(stream)))


def tgemm_debug_build() -> int:
    return int(load().tgemm_debug_build())


def tgemm_kernel_launches() -> int:
    return int(load().tgemm_kernel_launches())


def tgemm_version() -> int:
    return int(load().tgemm_version())


def tgemm_plan(mode: str, m: int, n: int, k: int, sm_count: int = 152, workspace: bool = True) -> dict:
    """The tensor-core tiles tgemm_tf32 (mode "tf32") or tgemm_bf16 (mode
    "bf16") would use; see tgemm_plan in include/tgemm.h."""
    out = (ctypes.c_int * 5)()
    st = load().tgemm_plan(1 if mode == "tf32" else 0, m, n, k, sm_count, 1 if workspace else 0, out)
    _check(st)
    return {"tile_rows": out[0], "tile_cols": out[1], "stream_k": bool(out[2]), "pieces": out[3],
            "pairs": bool(out[4])}


def tgemm_plan_f32(m: int, n: int, k: int, sm_count: int = 152) -> dict:
    """The 128 x 128 tiles tgemm_f32 would run; see tgemm_plan_f32 in include/tgemm.h."""
    out = (ctypes.c_int64 * 3)()
    _check(load().tgemm_plan_f32(m, n, k, sm_count, out))
    return {"whole_tiles": out[0], "split_tiles": out[1], "pieces": out[2]}


def raw(name: str):
    """The bare C function ``name`` (pointer-level calls, as a C caller makes them)."""
    return getattr(load(), name)
