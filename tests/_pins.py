"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each ``pin_*`` function takes a loaded oracle library (``oracle.load()`` or a
deliberately broken build of it) and raises ``AssertionError`` when the oracle
disagrees with the fact it is pinned to.  ``test_oracle_pins.py`` runs them on
the real oracle; ``test_oracle_mutants.py`` checks that every planted mistake
in the oracle's C source makes at least one of them fail.

The facts used: the pages' worked 4x4 example (fixture under ``golden/``),
identity and permutation matrices, closed forms (all-ones, rank-1, alternating
signs), exact rational brute force on tiny shapes, numpy's float64 matmul as a
library special case, exact integer inputs, and the pure-Python walk through
the pages' tiled algorithm.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np

import oracle
from oracle import tiled

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
U = 2.0 ** -53


def read_golden(name):
    """Parse a fixture of named integer matrices (``# comment`` lines skipped)."""
    mats, cur = {}, None
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.isalpha():
                cur = line
                mats[cur] = []
            else:
                mats[cur].append([int(v) for v in line.split()])
    return {k: np.array(v, dtype=np.float64) for k, v in mats.items()}


def gamma(k):
    """Higham's gamma_k = k u / (1 - k u): bound on |fl(sum) - sum| / sum |terms|."""
    return k * U / (1 - k * U)


def _rng(seed):
    return np.random.default_rng(seed)


def pin_worked_example(lib):
    g = read_golden("worked_4x4.txt")
    M, N, P_ref = g["M"], g["N"], g["P"]
    P, D = oracle.gemm(M, N, lib=lib)
    assert np.array_equal(P, P_ref), f"worked example: oracle {P} != fixture {P_ref}"
    assert np.array_equal(D, P_ref), "worked example: D must equal P for positive inputs"
    # The page's per-phase expressions for Block(0,0), TILE_WIDTH=2: phase 1 uses
    # k = 0, 1 and phase 2 uses k = 2, 3; P is their sum.
    Mi = [[int(v) for v in row] for row in M]
    Ni = [[int(v) for v in row] for row in N]
    for r in range(2):
        for c in range(2):
            ph1 = Mi[r][0] * Ni[0][c] + Mi[r][1] * Ni[1][c]
            ph2 = Mi[r][2] * Ni[2][c] + Mi[r][3] * Ni[3][c]
            assert P[r, c] == ph1 + ph2, f"Block(0,0) P({r},{c})"
    # Entry-wise path on the same fixture.
    rows, cols = np.nonzero(np.ones((4, 4)))
    Pe, De = oracle.gemm_entries(M, N, rows, cols, lib=lib)
    assert np.array_equal(Pe, P_ref[rows, cols]), "worked example (entries)"


def pin_identity(lib):
    rng = _rng(1)
    for (m, k, n) in [(5, 7, 3), (1, 9, 1), (16, 16, 16)]:
        M = rng.standard_normal((m, k))
        N = rng.standard_normal((k, n))
        P, D = oracle.gemm(M, np.eye(k), lib=lib)
        assert np.array_equal(P, M), f"M x I != M for {m}x{k}"
        assert np.array_equal(D, np.abs(M)), "D of M x I must be |M|"
        P, _ = oracle.gemm(np.eye(k), N, lib=lib)
        assert np.array_equal(P, N), f"I x N != N for {k}x{n}"


def pin_permutation(lib):
    rng = _rng(2)
    m, k = 6, 11
    M = rng.standard_normal((m, k))
    sigma = rng.permutation(k)                 # column j of P is column sigma[j] of M
    Pi = np.zeros((k, k))
    Pi[sigma, np.arange(k)] = 1.0
    P, _ = oracle.gemm(M, Pi, lib=lib)
    assert np.array_equal(P, M[:, sigma]), "M x permutation must permute the columns of M"
    P, _ = oracle.gemm(Pi.T, M.T.copy(), lib=lib)
    assert np.array_equal(P, M.T[sigma, :]), "permutation x N must permute the rows of N"


def pin_all_ones(lib):
    for (m, n, k) in [(3, 4, 5), (1, 1, 1), (7, 2, 300)]:
        P, D = oracle.gemm(np.ones((m, k)), np.ones((k, n)), lib=lib)
        assert np.all(P == k) and np.all(D == k), f"all-ones {m}x{n}x{k}: P must be k"


def pin_rank1(lib):
    for (m, n, k) in [(4, 6, 9), (9, 3, 2), (2, 5, 64)]:
        M = np.repeat(np.arange(1, m + 1, dtype=np.float64)[:, None], k, axis=1)
        N = np.repeat(np.arange(1, n + 1, dtype=np.float64)[None, :], k, axis=0)
        P, _ = oracle.gemm(M, N, lib=lib)
        expect = np.outer(np.arange(1, m + 1), np.arange(1, n + 1)) * k
        assert np.array_equal(P, expect), f"rank-1 closed form {m}x{n}x{k}"


def pin_alternating_signs(lib):
    # M(i,k) = (-1)^k (i+1), N(k,j) = j+1:  P = (i+1)(j+1) [K odd],  D = (i+1)(j+1) K.
    for (m, n, k) in [(3, 5, 6), (4, 2, 7)]:
        sgn = np.where(np.arange(k) % 2 == 0, 1.0, -1.0)
        M = np.outer(np.arange(1, m + 1), sgn)
        N = np.repeat(np.arange(1, n + 1, dtype=np.float64)[None, :], k, axis=0)
        P, D = oracle.gemm(M, N, lib=lib)
        base = np.outer(np.arange(1, m + 1), np.arange(1, n + 1)).astype(np.float64)
        assert np.array_equal(P, base * (k % 2)), f"alternating signs P {m}x{n}x{k}"
        assert np.array_equal(D, base * k), f"alternating signs D {m}x{n}x{k}"


def _exact(M, N):
    m, k = M.shape
    n = N.shape[1]
    Mf = [[Fraction(float(v)) for v in row] for row in M]
    Nf = [[Fraction(float(v)) for v in row] for row in N]
    P = [[sum((Mf[i][kk] * Nf[kk][j] for kk in range(k)), Fraction(0)) for j in range(n)]
         for i in range(m)]
    D = [[sum((abs(Mf[i][kk]) * abs(Nf[kk][j]) for kk in range(k)), Fraction(0)) for j in range(n)]
         for i in range(m)]
    return P, D


def pin_brute_force(lib):
    rng = _rng(3)
    shapes = [(m, n, k) for m in (1, 2, 3, 4) for n in (1, 2, 3, 4) for k in (1, 2, 3, 4)]
    shapes += [(7, 5, 6), (5, 7, 7), (2, 7, 3)]
    for (m, n, k) in shapes:
        # general doubles: the fp64 sum is within gamma_k * D of the exact sum
        M = rng.standard_normal((m, k)) * rng.choice([1.0, 1e3, 1e-3], size=(m, k))
        N = rng.standard_normal((k, n))
        P, D = oracle.gemm(M, N, lib=lib)
        Pe, De = _exact(M, N)
        for i in range(m):
            for j in range(n):
                err = abs(Fraction(float(P[i, j])) - Pe[i][j])
                assert err <= Fraction(gamma(k)) * De[i][j], f"brute force P({i},{j}) {m}x{n}x{k}"
                errd = abs(Fraction(float(D[i, j])) - De[i][j])
                assert errd <= Fraction(gamma(k)) * De[i][j], f"brute force D({i},{j}) {m}x{n}x{k}"
        # integers: exact
        Mi = rng.integers(-9, 10, size=(m, k)).astype(np.float64)
        Ni = rng.integers(-9, 10, size=(k, n)).astype(np.float64)
        P, D = oracle.gemm(Mi, Ni, lib=lib)
        Pe, De = _exact(Mi, Ni)
        assert all(P[i, j] == Pe[i][j] and D[i, j] == De[i][j] for i in range(m) for j in range(n)), \
            f"integer brute force {m}x{n}x{k}"
        rows = np.repeat(np.arange(m), n)
        cols = np.tile(np.arange(n), m)
        Pv, Dv = oracle.gemm_entries(Mi, Ni, rows, cols, lib=lib)
        assert all(Pv[c] == Pe[rows[c]][cols[c]] and Dv[c] == De[rows[c]][cols[c]]
                   for c in range(rows.size)), f"integer brute force (entries) {m}x{n}x{k}"


def pin_numpy(lib):
    rng = _rng(4)
    for (m, n, k) in [(37, 29, 53), (64, 1, 200), (1, 80, 3)]:
        M = rng.standard_normal((m, k))
        N = rng.standard_normal((k, n))
        P, D = oracle.gemm(M, N, lib=lib)
        Dn = np.abs(M) @ np.abs(N)
        bound = 2 * gamma(k) * Dn
        assert np.all(np.abs(P - M @ N) <= bound), f"numpy float64 matmul {m}x{n}x{k}"
        assert np.all(np.abs(D - Dn) <= bound), f"numpy |M||N| {m}x{n}x{k}"


def pin_dtypes(lib):
    rng = _rng(5)
    M32 = rng.standard_normal((9, 13)).astype(np.float32)
    N32 = rng.standard_normal((13, 6)).astype(np.float32)
    P32, D32 = oracle.gemm(M32, N32, lib=lib)
    P64, D64 = oracle.gemm(M32.astype(np.float64), N32.astype(np.float64), lib=lib)
    assert np.array_equal(P32, P64) and np.array_equal(D32, D64), "fp32 inputs must widen exactly"
    # bf16 bit patterns with known values: 0x3FC0 = 1.5, 0xC000 = -2.0, 0x3E80 = 0.25
    k = 37
    Mb = np.full((3, k), 0x3FC0, dtype=np.uint16)
    Nb = np.full((k, 4), 0xC000, dtype=np.uint16)
    P, D = oracle.gemm(Mb, Nb, lib=lib)
    assert np.all(P == -3.0 * k) and np.all(D == 3.0 * k), "bf16 1.5 x -2.0 closed form"
    Nq = np.full((k, 2), 0x3E80, dtype=np.uint16)
    P, _ = oracle.gemm(Mb, Nq, lib=lib)
    assert np.all(P == 0.375 * k), "bf16 1.5 x 0.25 closed form"
    # mixed storage: fp32 M with bf16 N equals the fp64 product of the decoded values
    Nd = np.full((13, 6), -2.0)
    Pm, _ = oracle.gemm(M32, np.full((13, 6), 0xC000, dtype=np.uint16), lib=lib)
    Pr, _ = oracle.gemm(M32.astype(np.float64), Nd, lib=lib)
    assert np.array_equal(Pm, Pr), "mixed fp32 x bf16"


def pin_entries_match_full(lib):
    rng = _rng(6)
    M = rng.standard_normal((23, 31))
    N = rng.standard_normal((31, 17))
    P, D = oracle.gemm(M, N, lib=lib)
    rows = rng.integers(0, 23, 50)
    cols = rng.integers(0, 17, 50)
    Pe, De = oracle.gemm_entries(M, N, rows, cols, lib=lib)
    # the same fp64 terms in the same ascending-k order: bit-identical
    assert np.array_equal(Pe, P[rows, cols]) and np.array_equal(De, D[rows, cols]), \
        "entry-wise and full oracle must agree bit for bit"


def pin_threads(lib):
    rng = _rng(7)
    M = rng.standard_normal((50, 40))
    N = rng.standard_normal((40, 30))
    ref = oracle.gemm(M, N, nthreads=1, lib=lib)
    for t in (2, 3, 7, 64):
        got = oracle.gemm(M, N, nthreads=t, lib=lib)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1]), f"threads={t}"


def pin_leading_dims(lib):
    rng = _rng(8)
    big_m = rng.standard_normal((12, 20))
    big_n = rng.standard_normal((15, 33))
    M = big_m[:, 3:18]       # 12 x 15, ld 20
    N = big_n[:, 5:14]       # 15 x 9, ld 33
    P, D = oracle.gemm(M, N, lib=lib)
    Pc, Dc = oracle.gemm(np.ascontiguousarray(M), np.ascontiguousarray(N), lib=lib)
    assert np.array_equal(P, Pc) and np.array_equal(D, Dc), "leading dimensions"
    Pe, _ = oracle.gemm_entries(M, N, [0, 11], [8, 0], lib=lib)
    assert np.array_equal(Pe, Pc[[0, 11], [8, 0]]), "leading dimensions (entries)"


def pin_empty(lib):
    P, D = oracle.gemm(np.zeros((0, 5)), np.zeros((5, 3)), lib=lib)
    assert P.shape == (0, 3)
    P, D = oracle.gemm(np.zeros((4, 0)), np.zeros((0, 3)), lib=lib)
    assert P.shape == (4, 3) and np.all(P == 0) and np.all(D == 0), "k = 0 is the empty sum"


def pin_tiled_walk(lib):
    rng = _rng(9)
    for (m, n, k, T) in [(4, 4, 4, 2), (6, 5, 7, 2), (9, 10, 11, 4), (8, 8, 8, 8), (5, 3, 13, 3)]:
        M = rng.integers(-5, 6, size=(m, k))
        N = rng.integers(-5, 6, size=(k, n))
        Pt, _, _ = tiled.tiled_product(M.tolist(), N.tolist(), T)
        P, _ = oracle.gemm(M.astype(np.float64), N.astype(np.float64), lib=lib)
        assert np.array_equal(P, np.array(Pt, dtype=np.float64)), f"tiled walk {m}x{n}x{k} T={T}"


def pin_transpose(lib):
    # element (i, j) of a 5 x 3 matrix holds 10 i + j: after transposing, element
    # (j, i) must hold 10 i + j; transposing twice is the identity.
    M = np.array([[10 * i + j for j in range(3)] for i in range(5)], dtype=np.float32)
    T = oracle.transpose(M)
    assert T.shape == (3, 5)
    assert all(T[j, i] == 10 * i + j for i in range(5) for j in range(3)), "transpose element map"
    assert np.array_equal(oracle.transpose(T), M), "transpose twice"
    assert oracle.transpose(np.zeros((0, 4))).shape == (4, 0)


PINS = [pin_worked_example, pin_identity, pin_permutation, pin_all_ones, pin_rank1,
        pin_alternating_signs, pin_brute_force, pin_numpy, pin_dtypes,
        pin_entries_match_full, pin_threads, pin_leading_dims, pin_empty, pin_tiled_walk, pin_transpose]


def failing_pins(lib):
    """Names of the pins that fail for ``lib`` (an empty list means all hold)."""
    failed = []
    for pin in PINS:
        try:
            pin(lib)
        except (AssertionError, RuntimeError, ValueError):
            failed.append(pin.__name__)
    return failed
