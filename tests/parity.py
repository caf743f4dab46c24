"""Helpers of the GPU parity tests: upload a case, run one entry point through
the C ABI, and compare with the oracle element by element.

Bars (from the error measure err = |C_gpu - P| / D with D = sum_k |M||N|):
  * integer-valued inputs whose partial sums are exact in fp32: C must equal
    the oracle exactly (float equality, so +0 == -0);
  * tgemm_f32 on general inputs: err <= 1e-5;
  * tgemm_tf32 / tgemm_bf16: err <= 4e-3.
Where D == 0 every term is zero, so C must be exactly 0 there.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from dense_tiled_matrix_gb300 import tgemm

TOL = {"f32": 1e-5, "tf32": 4e-3, "bf16": 4e-3}
ENTRY = {"f32": tgemm.tgemm_f32, "tf32": tgemm.tgemm_tf32, "bf16": tgemm.tgemm_bf16}


def to_device(arr: np.ndarray, device="cuda") -> torch.Tensor:
    """fp32 arrays as float32 tensors, uint16 bf16 bit patterns as bfloat16 tensors."""
    if arr.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr)).to(device)


def inputs_for(mode: str, case):
    """Host arrays in the storage type the entry point takes (bf16 rounds once, RNE)."""
    from dense_tiled_matrix_gb300 import inputs
    c = inputs.convert(case, "bf16" if mode == "bf16" else "f32")
    return c.A, c.B


def run(mode: str, A_host: np.ndarray, B_host: np.ndarray, C=None, device="cuda") -> torch.Tensor:
    A = to_device(A_host, device)
    B = to_device(B_host, device)
    out = ENTRY[mode](A, B, C)
    torch.cuda.synchronize()
    return out


def check(mode: str, got: np.ndarray, P: np.ndarray, D: np.ndarray, exact: bool, what: str = ""):
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == P.shape, f"{what}: shape {got.shape} != {P.shape}"
    assert np.all(np.isfinite(got)), f"{what}: non-finite outputs"
    if exact:
        ref = P.astype(np.float32).astype(np.float64)
        bad = np.argwhere(got != ref)
        assert bad.size == 0, (f"{what}: {len(bad)} of {got.size} elements differ from the exact result; "
                               f"first {bad[:3].tolist()} got {got[tuple(bad[0])]} want {ref[tuple(bad[0])]}")
        return 0.0
    diff = np.abs(got - P)
    zero = D == 0
    assert np.all(diff[zero] == 0), f"{what}: nonzero output where every term is zero"
    err = float(np.max(diff[~zero] / D[~zero])) if np.any(~zero) else 0.0
    assert err <= TOL[mode], f"{what}: max |C - P| / D = {err:.3e} > {TOL[mode]:.0e}"
    return err


def full_check(mode: str, case, what: str = ""):
    A, B = inputs_for(mode, case)
    P, D = oracle.gemm(A, B)
    C = run(mode, A, B).cpu().numpy()
    return check(mode, C, P, D, case.exact, what or f"{mode} {case}")
