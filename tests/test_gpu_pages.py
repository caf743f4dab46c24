"""The pages' naive and shared-memory tiled kernels (comparators) against the
oracle: fp32 FMA in ascending k, so integer inputs must be exact and random
inputs within the fp32 bound."""
import pytest
import torch

import oracle
from dense_tiled_matrix_gb300 import inputs, pages
import parity

pytestmark = pytest.mark.gpu

KERNELS = {
    "naive": lambda A, B: pages.tgemm_pages_naive_f32(A, B),
    "tiled16": lambda A, B: pages.tgemm_pages_tiled_f32(A, B, tile_width=16),
    "tiled32": lambda A, B: pages.tgemm_pages_tiled_f32(A, B, tile_width=32),
}


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    pages.load()


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("case", ["worked_4x4", "int64", "u128", "int1024", "edge"])
def test_pages_kernels(kernel, case):
    c = inputs.random_case(808, 133, 71, 45, kind="int") if case == "edge" else inputs.make(case)
    A, B = torch.from_numpy(c.A).cuda(), torch.from_numpy(c.B).cuda()
    C = KERNELS[kernel](A, B)
    torch.cuda.synchronize()
    P, D = oracle.gemm(c.A, c.B)
    parity.check("f32", C.cpu().numpy(), P, D, c.exact, f"pages {kernel} {c}")
