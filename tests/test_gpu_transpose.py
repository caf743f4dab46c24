"""Transpose kernels against the oracle's transpose, bit for bit: libtgemm's
tgemm_transpose_f32 (TMA form for matrices with 16-byte aligned bases and
pitches, padded 32 x 32 tiles otherwise) and the lecture's three kernels in
libtgemm_pages."""
import numpy as np
import pytest
import torch

import oracle
from dense_tiled_matrix_gb300 import inputs, pages, tgemm

pytestmark = pytest.mark.gpu

SHAPES = [(1, 1), (7, 5), (64, 32), (65, 33), (128, 96), (1000, 777), (1024, 1024), (2049, 3001)]
# Multiples of 4 in both dimensions (16-byte pitches: the TMA form) that are not
# multiples of its 128 x 32 input tile, so loads past the edge and clipped
# stores both occur; 4 x 8 is smaller than one tile.
ALIGNED_RAGGED = [(4, 8), (132, 36), (1000, 776), (2052, 3004), (128, 4100)]


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    tgemm.load()
    pages.load()


def _src(rows, cols, pad, seed):
    vals = inputs.uniform_pm1(seed, 0, (rows, cols + pad))
    store = torch.from_numpy(vals).cuda()
    return vals[:, :cols], store[:, :cols]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
@pytest.mark.parametrize("pad", [0, 1, 4])
def test_tgemm_transpose(shape, pad):
    rows, cols = shape
    host, src = _src(rows, cols, pad, 100 + rows + cols + pad)
    dst_store = torch.full((cols, rows + pad), float("nan"), device="cuda")
    dst = dst_store[:, :rows]
    tgemm.tgemm_transpose_f32(src, dst)
    torch.cuda.synchronize()
    assert np.array_equal(dst.cpu().numpy(), oracle.transpose(host))
    if pad:
        assert torch.all(torch.isnan(dst_store[:, rows:])), "wrote outside dst"


@pytest.mark.parametrize("shape", ALIGNED_RAGGED, ids=lambda s: f"{s[0]}x{s[1]}")
@pytest.mark.parametrize("pad", [0, 4, 8])
def test_tgemm_transpose_tma_edges(shape, pad):
    rows, cols = shape
    host, src = _src(rows, cols, pad, 300 + rows + cols + pad)
    dst_store = torch.full((cols, rows + pad), float("nan"), device="cuda")
    dst = dst_store[:, :rows]
    tgemm.tgemm_transpose_f32(src, dst)
    torch.cuda.synchronize()
    assert np.array_equal(dst.cpu().numpy(), oracle.transpose(host))
    if pad:
        assert torch.all(torch.isnan(dst_store[:, rows:])), "wrote outside dst"


@pytest.mark.parametrize("variant", sorted(pages.TRANSPOSE_VARIANTS))
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
def test_pages_transposes(variant, shape):
    rows, cols = shape
    host, src = _src(rows, cols, 3, 200 + rows + cols)
    dst = pages.tgemm_pages_transpose_f32(src, variant=variant)
    torch.cuda.synchronize()
    assert np.array_equal(dst.cpu().numpy(), oracle.transpose(host))


def test_transpose_argument_rules():
    src = torch.zeros((4, 4), device="cuda")
    lib = tgemm.load()
    ptr = src.data_ptr()
    assert lib.tgemm_transpose_f32(4, 4, ptr, 3, ptr + 4096, 4, None) == tgemm.TGEMM_ERR_INVALID_VALUE
    assert lib.tgemm_transpose_f32(4, 4, ptr, 4, ptr + 16, 4, None) == tgemm.TGEMM_ERR_INVALID_VALUE  # overlap
    assert lib.tgemm_transpose_f32(0, 4, None, 4, None, 1, None) == tgemm.TGEMM_OK
