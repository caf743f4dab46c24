"""The pages' tiled algorithm and its memory model, on the CPU.

hecess.blogspot.com "[Multi-Core & GPU Programming] CUDA - Matrix
Multiplication": "Work Flow" (which block/thread owns which P element),
"[Shared Memory]" (two phases of Block(0,0) in the 4x4, TILE_WIDTH=2 example)
and "Memory 분석" (global loads N^3 per operand naive, N^3/b tiled);
note.jhbae.stream "Lec 29 · GPU Architecture (2)" (2N^3 naive, 2N^2 (N/T)
tiled, 1/32 at TILE_WIDTH = 32).
"""
import numpy as np
import pytest

from oracle import tiled
import _pins


def test_block_thread_map_of_the_work_flow_section():
    # Block(0,1) in the page's notation is blockIdx.x = 1, blockIdx.y = 0: it owns
    # P(0,2), P(0,3), P(1,2), P(1,3).
    owned = {(r, c) for r in range(4) for c in range(4) if tiled.block_of(r, c, 2)[0] == (1, 0)}
    assert owned == {(0, 2), (0, 3), (1, 2), (1, 3)}
    owned = {(r, c) for r in range(4) for c in range(4) if tiled.block_of(r, c, 2)[0] == (0, 0)}
    assert owned == {(0, 0), (0, 1), (1, 0), (1, 1)}
    # col = blockIdx.x * blockDim.x + threadIdx.x, row = blockIdx.y * blockDim.y + threadIdx.y
    (bx, by), (tx, ty) = tiled.block_of(1, 3, 2)
    assert (bx * 2 + tx, by * 2 + ty) == (3, 1)


def test_two_phases_of_block_00():
    g = _pins.read_golden("worked_4x4.txt")
    M = g["M"].astype(int).tolist()
    N = g["N"].astype(int).tolist()
    P, _, phases = tiled.tiled_product(M, N, 2, record_block=(0, 0))
    assert len(phases) == 2
    for r in range(2):
        for c in range(2):
            assert phases[0][r][c] == M[r][0] * N[0][c] + M[r][1] * N[1][c]
            assert phases[1][r][c] == M[r][2] * N[2][c] + M[r][3] * N[3][c]
            assert P[r][c] == phases[0][r][c] + phases[1][r][c]
    assert np.array_equal(np.array(P), g["P"])


@pytest.mark.parametrize("n,b", [(4, 2), (8, 2), (8, 4), (12, 3), (16, 8), (32, 32)])
def test_global_load_counts(n, b):
    rng = np.random.default_rng(n * 100 + b)
    M = rng.integers(-3, 4, size=(n, n)).tolist()
    N = rng.integers(-3, 4, size=(n, n)).tolist()
    _, naive_loads = tiled.naive_product(M, N)
    P, tiled_loads, _ = tiled.tiled_product(M, N, b)
    assert naive_loads == 2 * n ** 3                       # 2N^3
    assert tiled_loads == 2 * n * n * (n // b)             # 2N^2 (N / TILE_WIDTH)
    assert tiled_loads * b == naive_loads                  # reduced by the tile width


def test_load_reduction_at_tile_width_32():
    n = 64
    M = np.ones((n, n), dtype=int).tolist()
    _, naive_loads = tiled.naive_product(M, M)
    _, tiled_loads, _ = tiled.tiled_product(M, M, 32)
    assert tiled_loads * 32 == naive_loads


def test_ragged_sizes_zero_fill():
    rng = np.random.default_rng(5)
    M = rng.integers(-3, 4, size=(5, 7)).tolist()
    N = rng.integers(-3, 4, size=(7, 3)).tolist()
    P, _, _ = tiled.tiled_product(M, N, 4)
    Pn, _ = tiled.naive_product(M, N)
    assert P == Pn
