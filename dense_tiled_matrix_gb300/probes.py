"""Python binding of libtgemm_probes: calibration kernels (read streams, the
paired-FMA rate; ``include/tgemm_probes.h``).  Argument marshalling only."""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtgemm_probes.so")

_I64, _VP = ctypes.c_int64, ctypes.c_void_p
SIGNATURES = {
    "tgemm_probe_read_tma": (ctypes.c_int, [_VP, _I64, _VP, _VP]),
    "tgemm_probe_read_ldg": (ctypes.c_int, [_VP, _I64, _VP, _VP]),
    "tgemm_probe_ffma2": (ctypes.c_int, [ctypes.c_int, _I64, _VP, _VP, _VP]),
}

_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise ImportError(f"libtgemm_probes.so not found at {path}; run dense_tiled_matrix_gb300.build.build()")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
        return _lib


def read_stream(buf, how: str, sum_out, stream=None) -> None:
    """Queue one probe over the whole of ``buf`` (a contiguous CUDA tensor);
    adds its 32-bit words into ``sum_out`` (a 1-element int64 CUDA tensor the
    caller zeroed).  ``how`` is "tma" or "ldg"."""
    import torch
    if not buf.is_contiguous() or not sum_out.is_cuda or sum_out.dtype != torch.int64:
        raise ValueError("read_stream: contiguous buf and an int64 CUDA sum")
    if stream is None:
        stream = torch.cuda.current_stream()
    fn = {"tma": load().tgemm_probe_read_tma, "ldg": load().tgemm_probe_read_ldg}[how]
    nbytes = buf.numel() * buf.element_size()
    rc = fn(buf.data_ptr() or None, nbytes, sum_out.data_ptr(), int(stream.cuda_stream))
    if rc != 0:
        raise RuntimeError(f"tgemm_probe_read_{how}: status {rc}")


def ffma2(warps_per_sm: int, iters: int, ab, out, stream=None) -> None:
    """Queue the paired-FMA probe: ``ab`` a 16-element float32 CUDA tensor
    (a[0..7], b[0..7]), ``out`` a 1-element float64 CUDA tensor the caller
    zeroed, which receives the sum of every thread's 64 accumulators."""
    import torch
    if ab.dtype != torch.float32 or ab.numel() != 16 or not ab.is_cuda or not ab.is_contiguous():
        raise ValueError("ffma2: ab must be 16 contiguous float32 on the GPU")
    if out.dtype != torch.float64 or not out.is_cuda:
        raise ValueError("ffma2: out must be a float64 CUDA tensor")
    if stream is None:
        stream = torch.cuda.current_stream()
    rc = load().tgemm_probe_ffma2(int(warps_per_sm), int(iters), ab.data_ptr(), out.data_ptr(),
                                  int(stream.cuda_stream))
    if rc != 0:
        raise RuntimeError(f"tgemm_probe_ffma2: status {rc}")
