"""NaN and infinity reach exactly the outputs they touch, on every path.

The pages define P(i,j) = sum_k M(i,k) N(k,j) and say nothing about special
values; the plainest reading is IEEE arithmetic, which the fp64 oracle
follows.  So a NaN in M(i, .) makes all of row i NaN, a NaN in N(., j) all of
column j, an infinity in N(k, j) makes P(i, j) an infinity of the sign of
M(i, k), or NaN where M(i, k) = 0 (0 * inf), and every other entry stays the
exact integer sum.  Split sums must keep this: the special values are placed
in the first and last k steps and in ragged edge columns, so that they sit in
different k-slices of the fp32 k-pieces, the tensor-core stream-K halves and
split-K pieces and the skinny kernel's cluster ranks, and in partial tiles.
"""
import numpy as np
import pytest
import torch

import oracle
from dense_tiled_matrix_gb300 import inputs
import parity

pytestmark = pytest.mark.gpu

BF16 = {"nan": 0x7FC0, "+inf": 0x7F80, "-inf": 0xFF80}
F32 = {"nan": np.float32(np.nan), "+inf": np.float32(np.inf), "-inf": np.float32(-np.inf)}


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def _plant(A, B, mode):
    val = BF16 if mode == "bf16" else F32
    m, k = A.shape
    n = B.shape[1]
    A[1, 3] = val["nan"]                     # row 1: NaN everywhere
    B[k // 2, n // 2] = val["nan"]           # column n / 2: NaN everywhere
    B[0, 2] = val["+inf"]                    # first k step, column 2: +-inf by sign of A[:, 0], NaN where 0
    B[k - 1, n - 1] = val["-inf"]            # last k step, last (ragged) column
    if m > 4:
        A[4, 0] = 0                          # 0 * inf = NaN at (4, 2)
        A[4, k - 1] = 0                      # and at (4, n - 1)


CASES = [
    ((64, 64, 64), ["f32", "tf32", "bf16"]),
    ((129, 257, 17), ["f32", "tf32", "bf16"]),        # ragged tiles everywhere
    ((1000, 900, 4100), ["f32"]),                      # fp32 k-pieces + ordered reduce
    ((2000, 2600, 1000), ["tf32", "bf16"]),            # tensor-core stream-K
    ((300, 520, 3100), ["tf32", "bf16"]),              # tensor-core split-K pieces
    ((16, 1000, 4100), ["bf16"]),                      # skinny, k split over a cluster
    ((33, 129, 70), ["bf16"]),                         # skinny 64-row form, ragged
]


@pytest.mark.parametrize("shape, modes", CASES, ids=lambda v: "x".join(map(str, v)) if isinstance(v, tuple) else "")
def test_nan_and_inf_propagate_like_the_oracle(shape, modes):
    m, n, k = shape
    for mode in modes:
        case = inputs.random_case(9000 + m + 3 * n + 7 * k, m, n, k, kind="int")
        A, B = parity.inputs_for(mode, case)
        A, B = A.copy(), B.copy()
        _plant(A, B, mode)
        C = parity.run(mode, A, B).cpu().numpy()
        P, _ = oracle.gemm(A, B)
        what = f"{mode} {shape}"
        assert np.array_equal(np.isnan(C), np.isnan(P)), what
        assert np.array_equal(np.isposinf(C), np.isposinf(P)), what
        assert np.array_equal(np.isneginf(C), np.isneginf(P)), what
        fin = np.isfinite(P)
        assert np.isnan(P).any() and np.isinf(P).any(), what   # the planted values reached the output
        assert np.array_equal(C[fin], P[fin].astype(np.float32)), what


def _bf16_bits(x):
    return (np.asarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


SUBNORMAL = [
    # label, a, b: every entry of A is a, of B is b, so every C entry is k a b;
    # a and b are exact in fp32, TF32 and bf16
    ("subnormal inputs", 2.0 ** -130, 1.0),          # a below 2^-126, result normal
    ("subnormal products", 2.0 ** -100, 2.0 ** -30),  # each product 2^-130, result normal
    ("subnormal results", 2.0 ** -130, 2.0 ** -15),   # result k 2^-145, below 2^-126
]


@pytest.mark.parametrize("shape", [(64, 64, 64), (16, 256, 64), (300, 520, 200)], ids=lambda s: "x".join(map(str, s)))
def test_subnormals(shape):
    """Subnormal operands, products and results are exact on every path (no
    flush to zero), as long as the operand itself is representable in the
    path's input format.  TF32 keeps the top 10 fraction bits of the fp32
    pattern, so an fp32 subnormal below 2^-136 (here 2^-140) reaches the
    tensor core as zero, while the FFMA path keeps it."""
    m, n, k = shape
    for label, a, b in SUBNORMAL:
        want = np.float32(np.float64(a) * np.float64(b) * k)
        for mode in ("f32", "tf32", "bf16"):
            A = np.full((m, k), a, np.float32)
            B = np.full((k, n), b, np.float32)
            if mode == "bf16":
                A, B = _bf16_bits(A), _bf16_bits(B)
            C = parity.run(mode, A, B).cpu().numpy()
            P, _ = oracle.gemm(A, B)
            assert np.array_equal(P.astype(np.float32), np.full((m, n), want)), (label, mode)   # the oracle, exact
            assert np.array_equal(C, np.full((m, n), want)), (label, mode, shape, float(C.min()), float(C.max()))
    # below TF32's window: FFMA exact, TF32 zero
    A = np.full((m, k), 2.0 ** -140, np.float32)
    B = np.ones((k, n), np.float32)
    want = np.float32(k * 2.0 ** -140)
    assert np.array_equal(parity.run("f32", A, B).cpu().numpy(), np.full((m, n), want))
    assert np.array_equal(parity.run("tf32", A, B).cpu().numpy(), np.zeros((m, n), np.float32))
