"""Pure-Python walk through the pages' tiled algorithm (test infrastructure).

Only the test suite uses this module.  It restates, for small exact (integer or
Fraction) inputs, the shared-memory tiled matrix multiply of hecess.blogspot.com
"[Multi-Core & GPU Programming] CUDA - Matrix Multiplication", section
"[Shared Memory]": the output is cut into TILE_WIDTH x TILE_WIDTH blocks
(block (bx, by) owns rows by*T.., columns bx*T..; section "Work Flow": x is the
column, y the row); each block walks the phases m = 0 .. ceil(K/T)-1; in a
phase every thread (tx, ty) copies one element of M and one of N into the
block's two shared tiles, the block synchronises, every thread adds the T
partial products of its row of subTileM and column of subTileN into its
private Pvalue, the block synchronises again; after the last phase each thread
stores its Pvalue once.

Where the pages assume Width is a multiple of TILE_WIDTH, this walk takes the
plainest reading for other sizes: a thread whose element lies outside M or N
stores 0 into the tile (and counts no global load), and a thread outside P
stores nothing.

It also counts global-memory element loads, to check the pages' load model
(section "Memory 분석" and the GT200 lecture summary: the naive kernel loads
2*N^3 elements, the tiled kernel 2*N^3/T).
"""
from __future__ import annotations


def naive_product(M, N):
    """One thread per output element reading M and N straight from global memory.

    Returns ``(P, loads)``; ``P`` is a list of rows of exact sums.
    """
    m, k = len(M), len(M[0]) if M else 0
    n = len(N[0]) if N else 0
    loads = 0
    P = [[0] * n for _ in range(m)]
    for row in range(m):
        for col in range(n):
            value = 0
            for kk in range(k):
                value += M[row][kk] * N[kk][col]
                loads += 2
            P[row][col] = value
    return P, loads


def tiled_product(M, N, tile, record_block=None):
    """The tiled kernel, block by block and phase by phase.

    ``record_block=(bx, by)`` additionally returns, for that block, the list of
    per-phase partial sums ``phases[p][ty][tx]`` (the bracketed groups of the
    page's Block(0,0) walk-through).

    Returns ``(P, loads, phases)``.
    """
    m = len(M)
    k = len(M[0]) if m else len(N)
    n = len(N[0]) if N else 0
    T = tile
    grid_x = -(-n // T)
    grid_y = -(-m // T)
    phases_count = -(-k // T)
    P = [[None] * n for _ in range(m)]
    loads = 0
    recorded = None
    for by in range(grid_y):
        for bx in range(grid_x):
            pvalue = [[0] * T for _ in range(T)]          # one register per thread
            block_phases = []
            for ph in range(phases_count):
                sub_m = [[0] * T for _ in range(T)]
                sub_n = [[0] * T for _ in range(T)]
                # every thread loads one element of each operand
                for ty in range(T):
                    for tx in range(T):
                        row = by * T + ty
                        col = bx * T + tx
                        mk = ph * T + tx
                        nk = ph * T + ty
                        if row < m and mk < k:
                            sub_m[ty][tx] = M[row][mk]
                            loads += 1
                        if nk < k and col < n:
                            sub_n[ty][tx] = N[nk][col]
                            loads += 1
                # (barrier) then every thread adds its T partial products
                partial = [[0] * T for _ in range(T)]
                for ty in range(T):
                    for tx in range(T):
                        s = 0
                        for kk in range(T):
                            s += sub_m[ty][kk] * sub_n[kk][tx]
                        partial[ty][tx] = s
                        pvalue[ty][tx] += s
                # (barrier) before the next phase overwrites the tiles
                block_phases.append(partial)
            for ty in range(T):
                for tx in range(T):
                    row = by * T + ty
                    col = bx * T + tx
                    if row < m and col < n:
                        P[row][col] = pvalue[ty][tx]
            if record_block == (bx, by):
                recorded = block_phases
    if m and n and k == 0:
        P = [[0] * n for _ in range(m)]
    return P, loads, recorded


def block_of(row, col, tile):
    """Block index (bx, by) and thread index (tx, ty) owning output P(row, col)."""
    return (col // tile, row // tile), (col % tile, row % tile)
