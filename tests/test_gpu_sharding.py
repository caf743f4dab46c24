"""Row sharding through libtgemm on the GPU.

P = M x N splits by rows with no communication (coffeejoa.com "CUDA.3 Writing
CUDA SIMT Kernels", "Cooperative Groups": work beyond one block, up to several
GPUs, as independent blocks of the output): shard r of W computes the row
block rows(m, W, r) of C from the same rows of A and the whole of B, each an
independent call of the C entry point.  Here every shard runs on the one GPU
the test has, one call after the other, exactly as it would on its own GPU;
the stitched C is compared element by element with the unsharded oracle
result: exactly on integer-valued inputs, within the path's bound otherwise.

The shards' row slices start at arbitrary rows, so some of them have base
addresses that TMA cannot take (bf16 rows of 1800 bytes); those operands go
through the library's re-pitch, and shards of at most 64 rows take the skinny
bf16 kernel.
"""
import numpy as np
import pytest
import torch

import oracle
from dense_tiled_matrix_gb300 import inputs, sharding
import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    from dense_tiled_matrix_gb300 import tgemm
    tgemm.load()
    yield
    assert tgemm.tgemm_get_device_status() == tgemm.TGEMM_OK


def _stitched(mode, A_host, B_host, world):
    A = parity.to_device(A_host)
    B = parity.to_device(B_host)
    blocks = []
    for rank in range(world):
        r0, r1, C_block = sharding.local_product(lambda a, b: parity.ENTRY[mode](a, b), A, B, world, rank)
        assert C_block.shape == (r1 - r0, B.shape[1])
        blocks.append(C_block)
    torch.cuda.synchronize()
    return torch.cat(blocks, dim=0).cpu().numpy()


@pytest.mark.parametrize("mode", ["f32", "tf32", "bf16"])
@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("shape", [(1001, 700, 900), (100, 2000, 1000), (4097, 301, 129)],
                         ids=lambda s: "x".join(map(str, s)))
def test_row_shards_stitch_to_the_oracle(mode, world, shape):
    m, n, k = shape
    for kind in ("int", "normal"):
        case = inputs.random_case(12000 + m + n + k + world, m, n, k, kind=kind)
        A_host, B_host = parity.inputs_for(mode, case)
        C = _stitched(mode, A_host, B_host, world)
        P, D = oracle.gemm(A_host, B_host)
        parity.check(mode, C, P, D, case.exact, f"{mode} {kind} {shape} in {world} row shards")


def test_row_shards_equal_the_unsharded_call_bit_for_bit():
    """Each C element's sum does not depend on which rows share its call for
    the fp32 FFMA path (one k-ascending FMA chain per element) when the shards
    keep whole tiles of the unsharded call's k-split plan: the shard of
    rows [0, 2048) and the unsharded product agree exactly on those rows."""
    m, n, k = 4096, 1024, 512
    case = inputs.random_case(12345, m, n, k, kind="normal")
    A = parity.to_device(case.A)
    B = parity.to_device(case.B)
    full = parity.ENTRY["f32"](A, B)
    half = parity.ENTRY["f32"](A[:2048], B)
    torch.cuda.synchronize()
    assert torch.equal(full[:2048], half)
