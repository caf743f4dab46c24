"""Schedules that fill the last wave, restated from the sources and checked on the CPU.

The pages' tiled algorithm (hecess.blogspot.com "[Multi-Core & GPU
Programming] CUDA - Matrix Multiplication", "Tiled Matrix Multiplication
Kernel") gives every output tile to one block, which walks all of its k
phases.  With T tiles on G = 152 SMs the last wave is partly empty (4096^3
fp32: 1024 tiles = 6 x 152 + 112).

* csrc/ffma_f32.cu (split remainder): the one-tile grid runs the 6 full
  rounds; the 112 tiles left are cut along k into `parts` pieces chosen to
  fill whole rounds best, each piece writes a partial tile to its workspace
  slot, and a reduce kernel adds a tile's pieces in part order.
* csrc/stream_k.cuh (tensor-core kernels): rounds of whole tiles b, b + G,
  ..., then the last G + r tiles flattened into (tile, k-phase) iterations
  cut into G equal runs; a tile split between two CTAs is finished by the one
  holding its first phases (head), which adds the other's partial (tail)
  after waiting for its flag.

Checked here: every iteration done once, every tile stored once, at most one
tail and one head per CTA, workspace slots in range, waits that cannot form a
cycle (co-residency comes from the cooperative launch), consecutive tiles in
each round, and, with exact integer data, that the partial sums add up to the
tile's sum.
"""
import numpy as np
import pytest

import launch_rules

BM, BN, BK = 128, 128, 16


def split_tail(m, n, k, G=152, stages=8):
    """(full-round tiles, remainder tiles, parts) of the fp32 launcher, or None."""
    tiles = -(-m // BM) * -(-n // BN)
    kt = -(-k // BK)
    r = tiles % G
    if r == 0 or 10 * r >= 9 * G:
        return None
    best, parts = 0.95, 1
    for s in range(2, 9):
        if kt // s < 2 * stages:
            break
        t = -(-(r * s) // G) / s
        if t < best:
            best, parts = t, s
    return None if parts == 1 else (tiles - r, r, parts)


def test_split_tail_choices():
    assert split_tail(4096, 4096, 4096) == (912, 112, 4)      # 112 x 4 quarters = 2.95 rounds
    assert split_tail(1024, 1024, 4096) == (0, 64, 7)          # less than one wave: all split
    assert split_tail(8192, 8192, 2048) is None                # 4096 tiles: last round 95 % full
    assert split_tail(4097, 3001, 1023) == (760, 32, 4)        # 792 tiles: 5 rounds + 32
    assert split_tail(8192, 8192, 512) is None                 # 4096 tiles: last round 95 % full
    assert split_tail(200, 150, 90) is None                    # 6 k-phases: too short to cut
    assert split_tail(256, 256, 65536) == (0, 4, 8)            # 4 tiles, 4096 phases: 8 pieces each
    for shape in [(2432, 2100, 2050), (1000, 900, 4100), (500, 20000, 2050), (2000, 2000, 4100)]:
        assert split_tail(*shape) is not None


@pytest.mark.parametrize("shape", [(4096, 4096, 4096), (2432, 2100, 2050), (1000, 900, 4100),
                                   (500, 20000, 2050), (3000, 6000, 4096), (4097, 3001, 1023), (1000, 700, 900)])
def test_split_tail_covers_every_phase_once(shape):
    m, n, k = shape
    full, rest, parts = split_tail(m, n, k)
    kt = -(-k // BK)
    assert kt // parts >= 16
    tiles = full + rest
    done = np.zeros((tiles, kt), dtype=np.int64)
    done[:full] += 1                                           # one-tile grid: blocks 0 .. full-1
    for u in range(rest * parts):                              # split kernel: block u -> slot u
        t, part = full + u // parts, u % parts
        k0, k1 = kt * part // parts, kt * (part + 1) // parts
        assert k1 - k0 >= 16
        done[t, k0:k1] += 1
    assert (done == 1).all()
    # reduce block b reads slots b * parts .. b * parts + parts - 1, all written
    assert {b * parts + q for b in range(rest) for q in range(parts)} == set(range(rest * parts))


def test_split_tail_sums_exactly_on_integers():
    rng = np.random.default_rng(3)
    k, parts = 160, 3
    kt = k // BK
    A = rng.integers(-8, 9, size=(BM, k)).astype(np.float32)
    B = rng.integers(-8, 9, size=(k, BN)).astype(np.float32)
    slots = [A[:, kt * q // parts * BK:kt * (q + 1) // parts * BK] @ B[kt * q // parts * BK:kt * (q + 1) // parts * BK]
             for q in range(parts)]
    C = np.zeros((BM, BN), dtype=np.float32)
    for q in range(parts):                                     # part order, as the reduce kernel
        C += slots[q]
    np.testing.assert_array_equal(C, A @ B)


def plan(tiles, kt, b, grid):
    """(whole tiles, first stream-K tile, run start, run end) of CTA b."""
    rounds, r = divmod(tiles, grid)
    tiles_sk = 0
    if r > 0 and rounds >= 1 and r * kt >= grid:
        tiles_sk, rounds, r = grid + r, rounds - 1, 0
    n_dp = rounds + (1 if b < r else 0)
    total = tiles_sk * kt
    return n_dp, tiles - tiles_sk, total * b // grid, total * (b + 1) // grid


def segments_of(tiles, kt, grid):
    """Per CTA, its segments (tile, first k-phase, end k-phase), in its own order."""
    out = []
    for b in range(grid):
        n_dp, t_sk0, v, v1 = plan(tiles, kt, b, grid)
        segs = [(b + j * grid, 0, kt) for j in range(n_dp)]
        while v < v1:
            q, ka = divmod(v, kt)
            kz = min(kt, ka + (v1 - v))
            segs.append((t_sk0 + q, ka, kz))
            v += kz - ka
        out.append(segs)
    return out


def roles(segs, kt):
    """'store' for a whole tile, 'tail' (writes ws[b], raises flag b), 'head' (waits for flag b+1)."""
    r = []
    for (_, ka, kz) in segs:
        if ka == 0 and kz == kt:
            r.append("store")
        elif ka > 0:
            r.append("tail")
        else:
            r.append("head")
    return r


# (tiles, KT) of persistent tensor-core launches: 256 x 256 tiles (KT for
# 128 bytes of k per phase) and some that leave a partial last wave.
PLANS = [(256, 128), (1024, 128), (156, 49), (176, 16), (198, 65), (628, 129), (304, 64), (153, 128)]


@pytest.mark.parametrize("sm_count", [152, 148, 132])
@pytest.mark.parametrize("tiles,kt", PLANS)
def test_schedule_invariants(tiles, kt, sm_count):
    per_cta = segments_of(tiles, kt, sm_count)
    done = np.zeros((tiles, kt), dtype=np.int64)
    stores = np.zeros(tiles, dtype=np.int64)
    for b, segs in enumerate(per_cta):
        rs = roles(segs, kt)
        n_dp = plan(tiles, kt, b, sm_count)[0]
        assert rs[:n_dp] == ["store"] * n_dp
        assert rs.count("tail") <= 1 and rs.count("head") <= 1
        if "tail" in rs:
            assert rs.index("tail") == n_dp                   # first stream-K segment: before any wait
        if "head" in rs:
            assert rs.index("head") == len(rs) - 1            # its only wait is its last segment
            assert b + 1 < sm_count                           # ws slot and flag of CTA b + 1 exist
            t, ka, kz = segs[-1]
            partner = per_cta[b + 1][plan(tiles, kt, b + 1, sm_count)[0]]
            assert partner == (t, kz, kt)                     # CTA b+1's first stream-K segment
        for (t, ka, kz), role in zip(segs, rs):
            done[t, ka:kz] += 1
            if role != "tail":
                stores[t] += 1
    assert (done == 1).all()
    assert (stores == 1).all()
    # Round j of whole tiles: the CTAs hold G consecutive tiles (L2 reuse as in the plain grid).
    n_dp0 = plan(tiles, kt, 0, sm_count)[0]
    for j in range(n_dp0):
        held = sorted(per_cta[b][j][0] for b in range(sm_count) if j < plan(tiles, kt, b, sm_count)[0])
        assert held == list(range(held[0], held[0] + len(held)))


def test_plan_regions():
    G = 152
    assert plan(1024, 256, 0, G)[:2] == (5, 1024 - 264)       # 5 rounds, then 264 tiles stream-K
    assert plan(152, 132, 7, G) == (1, 152, 0, 0)             # r = 0: whole tiles only
    assert plan(153, 128, 0, G)[:2] == (2, 153) and plan(153, 128, 1, G)[0] == 1   # r KT < G


def test_head_plus_tail_is_the_full_sum_on_integers():
    # A scaled-down grid runs the same schedule: 5 x 3 tiles on 4 CTAs = two
    # rounds of whole tiles, then 7 tiles cut into 4 stream-K runs.
    rng = np.random.default_rng(7)
    m, n, k, grid = 600, 260, 96, 4
    kt = k // BK
    tiles_m = -(-m // BM)
    tiles = tiles_m * -(-n // BN)
    per_cta = segments_of(tiles, kt, grid)
    assert plan(tiles, kt, 0, grid)[:2] == (2, 8)
    assert sum(roles(s, kt).count("head") for s in per_cta) == grid - 1
    A = rng.integers(-8, 9, size=(m, k)).astype(np.float32)
    B = rng.integers(-8, 9, size=(k, n)).astype(np.float32)
    C = np.full((m, n), np.nan, dtype=np.float32)
    ws = {}
    for b in reversed(range(grid)):       # tails of higher CTAs first: the order the flags enforce
        for (t, ka, kz), role in zip(per_cta[b], roles(per_cta[b], kt)):
            tm, tn = t % tiles_m, t // tiles_m     # any bijection serves the check
            r0, c0 = tm * BM, tn * BN
            part = A[r0:r0 + BM, ka * BK:kz * BK] @ B[ka * BK:kz * BK, c0:c0 + BN]
            if role == "tail":
                ws[b] = part
            else:
                if role == "head":
                    part = part + ws[b + 1]
                C[r0:r0 + BM, c0:c0 + BN] = part
    assert not np.isnan(C).any()
    np.testing.assert_array_equal(C, A @ B)


# ---- tcgen05 kernels (csrc/umma.cu): tile width, then the same plan ----
def umma_choice(m, n, k, mode, G=152):
    """(tile width, tiles, KT, stream-K) the launcher picks: 256 x BN or 128 x
    BN tiles by the rule of launch_rules.tile_rows.  Stream-K (always with BN =
    256) when the plan has a region and whole tiles would fill less than 3/4
    of the occupied CTA slots; otherwise TF32 takes BN = 224 when that fills
    them better by more than 2 %."""
    bm = launch_rules.tile_rows(m, n, k, mode, G)
    kt = launch_rules.k_phases(k, mode)
    tiles = launch_rules.tiles_of(m, n, bm)
    if launch_rules.stream_k(tiles, kt, G):
        return 256, tiles, kt, True
    fill = lambda bn: launch_rules.slot_fill(m, n, bm, bn, G)
    bn = 224 if mode == "tf32" and fill(224) > 1.02 * fill(256) else 256
    return bn, launch_rules.tiles_of(m, n, bm, bn), kt, False


def test_umma_choices_on_the_benchmarked_shapes():
    assert umma_choice(4096, 4096, 4096, "tf32") == (224, 304, 128, False)   # 2 full waves
    assert umma_choice(8192, 8192, 8192, "bf16")[::3] == (256, False)        # 1024 tiles: 96 % filled
    assert umma_choice(4097, 3001, 1023, "tf32")[0] == 256


@pytest.mark.parametrize("mode", ["tf32", "bf16"])
def test_umma_tile_rows_on_measured_shapes(mode):
    """The tile-height rule on the shapes whose timings chose it: wide tiles at
    long k, and at 1024 <= k < 3072 where their rounds are at least as full
    (measured faster or equal); 128-row tiles where the wide rounds are
    emptier (1536 x 9728 x 1024: 3/4 of two rounds against three full ones),
    too few (2048^3: 64 wide tiles) or split (4097 x 3001 x 1023), and at k < 1024."""
    for shape in [(8192, 8192, 8192), (8192, 8192, 1024), (2048, 4864, 1024), (2048, 4864, 2048),
                  (3000, 6000, 1024), (2900, 5000, 1030), (4096, 4096, 2048), (6144, 3072, 1024)]:
        assert launch_rules.tile_rows(*shape, mode) == 256, shape
    for shape in [(1536, 9728, 1024), (2048, 2048, 2048), (4097, 3001, 1023), (2000, 2600, 1000),
                  (8192, 8192, 1000), (2000, 4800, 999)]:
        assert launch_rules.tile_rows(*shape, mode) == 128, shape
    # the two grids' slot fills on the deciding shapes
    assert launch_rules.slot_fill(1536, 9728, 256) == 0.75 and launch_rules.slot_fill(1536, 9728, 128) == 1.0
    assert launch_rules.slot_fill(2900, 5000, 256) == launch_rules.slot_fill(2900, 5000, 128)


def test_umma_pieces_choices():
    """Split-K pieces where the tiles fill less than one round: as many pieces
    as fit in the round, each at least 8 k-phases; none at a round or more,
    nor where pieces would be shorter."""
    P = launch_rules.pieces
    assert P(1024, 1024, 8192, "bf16") == 9 and P(1024, 1024, 8192, "tf32") == 9   # 16 wide tiles
    assert P(256, 256, 65536, "bf16") == 128 and P(256, 256, 65536, "tf32") == 152  # one tile
    assert P(300, 520, 3100, "bf16") == 6                                          # 6 tiles, 49 phases
    assert P(65, 4096, 4096, "bf16") == 8                                          # 16 tiles, 64 phases
    assert P(1000, 1001, 2000, "bf16") == 4                                        # 32 128-row tiles
    assert P(2048, 2048, 1024, "bf16") == 0          # 128 tiles: 152 // 128 = 1
    assert P(4096, 4096, 4096, "bf16") == 0          # a full round and more
    assert P(1024, 1024, 512, "bf16") == 0           # 8 phases: no two pieces of 8
    assert P(1024, 1024, 512, "tf32") == 2           # 16 TF32 phases


@pytest.mark.parametrize("shape", [(1024, 1024, 8192), (300, 520, 3100), (256, 256, 65536), (1000, 1001, 2000)])
def test_umma_pieces_cover_k_once_and_sum_exactly(shape):
    """Piece p of a tile takes k-phases [KT p / P, KT (p + 1) / P): together they
    cover every phase once, none is empty, and their partial sums added in
    piece order give the tile's sum exactly on integers."""
    m, n, k = shape
    for mode in ("bf16", "tf32"):
        pc = launch_rules.pieces(m, n, k, mode)
        kt = launch_rules.k_phases(k, mode)
        ranges = [(kt * p // pc, kt * (p + 1) // pc) for p in range(pc)]
        assert ranges[0][0] == 0 and ranges[-1][1] == kt
        assert all(a < b and b - a >= 8 for a, b in ranges)
        assert all(ranges[i][1] == ranges[i + 1][0] for i in range(pc - 1))
    rng = np.random.default_rng(7)
    bk = 64
    A = rng.integers(-3, 4, (16, k)).astype(np.float32)
    B = rng.integers(-3, 4, (k, 8)).astype(np.float32)
    kt = launch_rules.k_phases(k, "bf16")
    pc = launch_rules.pieces(m, n, k, "bf16")
    C = np.zeros((16, 8), np.float32)
    for p in range(pc):
        a, b = kt * p // pc * bk, min(k, kt * (p + 1) // pc * bk)
        C += A[:, a:b] @ B[a:b]
    np.testing.assert_array_equal(C, A @ B)


@pytest.mark.parametrize("mode", ["tf32", "bf16"])
def test_umma_stream_k_shapes(mode):
    G = 152
    # the GPU parity shapes for the split path: wide with no whole-tile round,
    # narrow, wide with a round
    for shape in [(3300, 3000, 3100), (2000, 2600, 1000), (2600, 4000, 4100)]:
        bn, tiles, kt, sk = umma_choice(*shape, mode)
        assert sk, shape
        per_cta = segments_of(tiles, kt, G)
        assert sum(roles(s, kt).count("head") for s in per_cta) > 20
    assert not umma_choice(1024, 1024, 1024, mode)[3]   # fewer tiles than SMs


# ---- split-K pieces of the tcgen05 kernels: slot layout and reduce, simulated ----
def _slot_of(part, bm, bn):
    """A piece's partial tile (bm x bn) in the workspace slot layout the
    epilogue writes: float4 ((h * bn/32 + c) * 8 + q) * 128 + r = columns
    32c + 4q .. +3 of row 128h + r."""
    slot = np.empty((bm * bn // 4, 4), np.float32)
    for h in range(bm // 128):
        for c in range(bn // 32):
            for q in range(8):
                f0 = ((h * (bn // 32) + c) * 8 + q) * 128
                slot[f0:f0 + 128] = part[128 * h:128 * h + 128, 32 * c + 4 * q:32 * c + 4 * q + 4]
    return slot


def _reduce(slots, tiles_m, tiles_n, M, N, bm, bn, group_m, pieces):
    """umma_pieces_reduce_kernel's index arithmetic: block (t, j), thread i,
    float4 f = 1024 j + 256 r + i; the pieces added in order; rows and columns
    past C skipped.  Returns C and how often each element was written."""
    C = np.full((M, N), np.nan, np.float32)
    writes = np.zeros((M, N), np.int64)
    k4 = bm * bn // 4
    for t in range(tiles_m * tiles_n):
        per_group = group_m * tiles_n
        g, first = t // per_group, (t // per_group) * group_m
        rows_g = min(tiles_m - first, group_m)
        tm, tn = first + (t - g * per_group) % rows_g, (t - g * per_group) // rows_g
        v = slots[t * pieces].copy()
        for p in range(1, pieces):
            v += slots[t * pieces + p]
        for f in range(k4):
            gq = f >> 7
            q, hc = gq & 7, gq >> 3
            row = tm * bm + (hc // (bn // 32)) * 128 + (f & 127)
            col = tn * bn + (hc % (bn // 32)) * 32 + q * 4
            if row >= M:
                continue
            for j in range(4):
                if col + j < N:
                    C[row, col + j] = v[f, j]
                    writes[row, col + j] += 1
    return C, writes


@pytest.mark.parametrize("bm, M, N, group_m", [(256, 300, 520, 8), (128, 257, 300, 16)])
def test_split_k_pieces_slot_layout_and_reduce(bm, M, N, group_m):
    """The pieces of every tile, stored in the epilogue's slot layout and added
    by the reduce's index map in piece order, give A @ B exactly (integer
    inputs), with every element of C written once and nothing outside it."""
    bn, bk, pieces = 256, 64, 3
    K = 5 * bk + 17                                   # ragged k: the last phase partly zero-filled
    rng = np.random.default_rng(3)
    A = rng.integers(-3, 4, (M, K)).astype(np.float32)
    B = rng.integers(-3, 4, (K, N)).astype(np.float32)
    tiles_m, tiles_n = -(-M // bm), -(-N // bn)
    kt = -(-K // bk)
    Ap = np.zeros((tiles_m * bm, kt * bk), np.float32)
    Ap[:M, :K] = A
    Bp = np.zeros((kt * bk, tiles_n * bn), np.float32)
    Bp[:K, :N] = B
    slots = []
    for t in range(tiles_m * tiles_n):
        per_group = group_m * tiles_n
        g, first = t // per_group, (t // per_group) * group_m
        rows_g = min(tiles_m - first, group_m)
        tm, tn = first + (t - g * per_group) % rows_g, (t - g * per_group) // rows_g
        for p in range(pieces):
            ka, kz = kt * p // pieces * bk, kt * (p + 1) // pieces * bk
            part = Ap[tm * bm:(tm + 1) * bm, ka:kz] @ Bp[ka:kz, tn * bn:(tn + 1) * bn]
            slots.append(_slot_of(part, bm, bn))
    C, writes = _reduce(slots, tiles_m, tiles_n, M, N, bm, bn, group_m, pieces)
    assert np.array_equal(writes, np.ones((M, N), np.int64))
    np.testing.assert_array_equal(C, A @ B)
