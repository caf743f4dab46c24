"""tgemm_tf32_noalloc: the TF32 product for callers that cannot let the library
allocate device memory (their memory is owned by their own allocator or a
fixed arena, or their hot path must not allocate).  Its scratch lives in a
static device array of TGEMM_NOALLOC_SCRATCH_BYTES instead.

The test calls the entry point through the C ABI twice in a row, with
different shapes (the second needs a re-pitched A as well as the transposed B,
so it reuses the array the first call wrote), and checks each output element
by element against the CPU oracle (hecess.blogspot.com "[Multi-Core & GPU
Programming] CUDA - Matrix Multiplication", section "[Matrix
Multiplication]": P(i,j) = sum_k M(i,k) N(k,j)):
  * integer-valued inputs whose sums are exact in fp32 must match exactly;
  * N(0,1) inputs within the TF32 bound max |C - P| / (|A| |B|) <= 4e-3.
As an extra check the output is also compared with tgemm_tf32 on the same
inputs.  A shape too large for the array must be refused before any work is
queued.

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


def _run(name, case, a_pad):
    """C from entry point `name` with A stored at a leading dimension of k + a_pad
    (a_pad = 1 makes lda * 4 not a multiple of 16, so A is re-pitched)."""
    m, n, k = case.m, case.n, case.k
    A_store = torch.zeros((m, k + a_pad), dtype=torch.float32, device="cuda")
    A_store[:, :k] = torch.from_numpy(case.A).cuda()
    A = A_store[:, :k]
    B = torch.from_numpy(case.B).cuda()
    C = torch.full((m, n), float("nan"), device="cuda")
    status = _raw_call(name, A, B, C, k + a_pad)
    assert status == tgemm.TGEMM_OK, f"{name}: {tgemm.tgemm_status_string(status)}: {tgemm.tgemm_last_error()}"
    torch.cuda.synchronize()
    return C.cpu().numpy().astype(np.float64)


def _check_against_oracle(m, n, k, seed, a_pad, kind):
    case = inputs.random_case(seed, m, n, k, kind=kind)
    got = _run("tgemm_tf32_noalloc", case, a_pad)
    P, D = oracle.gemm(case.A, case.B)
    assert np.all(np.isfinite(got)), "non-finite output"
    if case.exact:
        ref = P.astype(np.float32).astype(np.float64)
        bad = np.argwhere(got != ref)
        assert bad.size == 0, f"{len(bad)} elements differ from the oracle's exact sums, first {bad[:3].tolist()}"
    else:
        diff = np.abs(got - P)
        zero = D == 0
        assert np.all(diff[zero] == 0)
        err = float(np.max(diff[~zero] / D[~zero]))
        assert err <= TOL_TF32, f"tgemm_tf32_noalloc vs oracle: {err:.3e}"
    # extra check: the allocating entry point agrees within the same bound
    other = _run("tgemm_tf32", case, a_pad)
    err_other = float(np.max(np.abs(got - other) / np.where(D == 0, 1.0, D)))
    assert err_other <= TOL_TF32, f"tgemm_tf32_noalloc vs tgemm_tf32: {err_other:.3e}"


@pytest.mark.parametrize("kind", ["int", "normal"])
def test_noalloc_matches_oracle_on_two_calls_in_a_row(kind):
    base = 9001 if kind == "int" else 9101
    _check_against_oracle(1000, 700, 900, seed=base, a_pad=0, kind=kind)     # transposed B in the array
    _check_against_oracle(333, 517, 301, seed=base + 1, a_pad=1, kind=kind)  # re-pitched A and transposed B
    assert tgemm.tgemm_get_device_status() == tgemm.TGEMM_OK


def test_noalloc_refuses_shapes_beyond_its_array():
    n = k = 4096                                        # B^T alone needs 64 MiB > 32 MiB
    A = torch.zeros((8, k), device="cuda")
    B = torch.zeros((k, n), device="cuda")
    C = torch.zeros((8, n), device="cuda")
    status = _raw_call("tgemm_tf32_noalloc", A, B, C, k)
    assert status == tgemm.TGEMM_ERR_INVALID_VALUE
    assert "TGEMM_NOALLOC_SCRATCH_BYTES" in tgemm.tgemm_last_error()
