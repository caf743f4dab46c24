"""tgemm_tf32_noalloc: the TF32 product for callers that cannot let the library
allocate device memory (their memory is owned by their own allocator or a
fixed arena, or their hot path must not allocate).  Its scratch lives in a
static device array of TGEMM_NOALLOC_SCRATCH_BYTES instead.

The test calls the entry point through the C ABI twice in a row, with
different shapes (the second needs a re-pitched A as well as the transposed B,
so it reuses the array the first call wrote), and checks each output against
tgemm_tf32 on the same inputs, within the TF32 bound the other parity tests
use: max |C_noalloc - C_tf32| / (|A| |B|) <= 4e-3.  It also checks that a
shape too large for the array is refused before any work is queued.

This file is named so that pytest collects it last; it passes alone in a fresh
process and after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from dense_tiled_matrix_gb300 import inputs, tgemm

pytestmark = pytest.mark.gpu

TOL_TF32 = 4e-3


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    tgemm.load()


def _raw_call(name, A, B, C, lda):
    """Pointer-level call of the C entry point, as a C caller makes it."""
    fn = tgemm.raw(name)
    m, k = A.shape[0], B.shape[0]
    n = B.shape[1]
    stream = torch.cuda.current_stream().cuda_stream
    return fn(m, n, k, ctypes.c_void_p(A.data_ptr()), lda, ctypes.c_void_p(B.data_ptr()), B.stride(0),
              ctypes.c_void_p(C.data_ptr()), C.stride(0), ctypes.c_void_p(stream))


def _compare(m, n, k, seed, a_pad):
    case = inputs.random_case(seed, m, n, k, kind="normal")
    # A with a leading dimension of k + a_pad (a_pad = 1 makes lda*4 not a multiple of 16)
    A_store = torch.zeros((m, k + a_pad), dtype=torch.float32, device="cuda")
    A_store[:, :k] = torch.from_numpy(case.A).cuda()
    A = A_store[:, :k]
    B = torch.from_numpy(case.B).cuda()
    C_ref = torch.full((m, n), float("nan"), device="cuda")
    C_new = torch.full((m, n), float("nan"), device="cuda")
    assert _raw_call("tgemm_tf32", A, B, C_ref, k + a_pad) == tgemm.TGEMM_OK, tgemm.tgemm_last_error()
    assert _raw_call("tgemm_tf32_noalloc", A, B, C_new, k + a_pad) == tgemm.TGEMM_OK, tgemm.tgemm_last_error()
    torch.cuda.synchronize()
    _, D = oracle.gemm(case.A, case.B)
    diff = np.abs(C_new.cpu().numpy().astype(np.float64) - C_ref.cpu().numpy().astype(np.float64))
    assert np.all(np.isfinite(diff)), "non-finite output"
    err = float(np.max(diff / D))
    assert err <= TOL_TF32, f"tgemm_tf32_noalloc vs tgemm_tf32: {err:.3e}"


def test_noalloc_matches_tgemm_tf32_on_two_calls_in_a_row():
    _compare(1000, 700, 900, seed=9001, a_pad=0)     # transposed B in the array
    _compare(333, 517, 301, seed=9002, a_pad=1)      # re-pitched A and transposed B
    assert tgemm.tgemm_get_device_status() == tgemm.TGEMM_OK


def test_noalloc_refuses_shapes_beyond_its_array():
    n = k = 4096                                        # B^T alone needs 64 MiB > 32 MiB
    A = torch.zeros((8, k), device="cuda")
    B = torch.zeros((k, n), device="cuda")
    C = torch.zeros((8, n), device="cuda")
    status = _raw_call("tgemm_tf32_noalloc", A, B, C, k)
    assert status == tgemm.TGEMM_ERR_INVALID_VALUE
    assert "TGEMM_NOALLOC_SCRATCH_BYTES" in tgemm.tgemm_last_error()
