"""The fp32 kernel's persistent schedule, restated from csrc/ffma_f32.cu and checked on the CPU.

The pages' tiled algorithm (hecess.blogspot.com "[Multi-Core & GPU
Programming] CUDA - Matrix Multiplication", "Tiled Matrix Multiplication
Kernel") gives every output tile to one block, which walks all of its k
phases.  With 1024 tiles of 128 x 128 on 152 SMs that leaves a last wave of
112 tiles (0.74 of a wave).  The persistent form runs one CTA per SM: with
T = q G + r tiles on G CTAs, CTA b first takes whole tiles b, b + G, ... for
q - 1 rounds (G consecutive tiles in flight, as in the one-tile-per-block
grid), then the last G + r tiles are flattened into (tile, k-phase)
iterations and cut into G equal runs ("stream-K").  A tile whose phases fall
to two CTAs is finished by the one holding its first phases (the head), which
adds the other's partial sums (the tail) after waiting for its flag.  With
r = 0, or r KT < G, there is no stream-K region.

Checked here: every iteration done once, every C tile stored once, at most one
tail and one head per CTA, workspace slots in range, waits that cannot form a
cycle (co-residency comes from the cooperative launch), consecutive tiles in
each round, and, with exact integer data, head + tail equals the tile's sum.
"""
import numpy as np
import pytest

BM, BN, BK = 128, 128, 16


def selected(m, n, k, sm_count, short_k=2048):
    """The launcher's rule: long k, and the one-tile-per-block grid would leave
    at least a tenth of its block slots empty, and there is a stream-K region."""
    tiles = -(-m // BM) * -(-n // BN)
    kt = -(-k // BK)
    rounds, r = divmod(tiles, sm_count)
    waves = -(-tiles // sm_count)
    return k >= short_k and rounds >= 1 and r > 0 and r * kt >= sm_count and 10 * tiles < 9 * waves * sm_count


def plan(tiles, kt, b, grid):
    """(whole tiles, first stream-K tile, run start, run end) of CTA b."""
    rounds, r = divmod(tiles, grid)
    tiles_sk = 0
    if r > 0 and rounds >= 1 and r * kt >= grid:
        tiles_sk, rounds, r = grid + r, rounds - 1, 0
    n_dp = rounds + (1 if b < r else 0)
    total = tiles_sk * kt
    return n_dp, tiles - tiles_sk, total * b // grid, total * (b + 1) // grid


def segments(m, n, k, grid):
    """Per CTA, its segments (tile, first k-phase, end k-phase), in its own order."""
    tiles = -(-m // BM) * -(-n // BN)
    kt = -(-k // BK)
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
    return out, tiles, kt


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


SHAPES = [(4096, 4096, 4096), (4097, 3001, 2048), (8192, 8192, 2048), (3000, 6000, 4096),
          (4096, 4096, 8192), (2432, 1000, 2100), (2100, 1100, 2048), (2000, 2000, 4096)]


@pytest.mark.parametrize("sm_count", [152, 148, 132])
@pytest.mark.parametrize("shape", SHAPES)
def test_schedule_invariants(shape, sm_count):
    m, n, k = shape
    per_cta, tiles, kt = segments(m, n, k, sm_count)
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
        held = sorted(per_cta[b][j][0] for b in range(sm_count) if len(per_cta[b]) > j
                      and roles(per_cta[b], kt)[j] == "store" and j < plan(tiles, kt, b, sm_count)[0])
        assert held == list(range(held[0], held[0] + len(held)))


def test_selection_and_regions():
    G = 152
    assert plan(1024, 256, 0, G)[:2] == (5, 1024 - 264)       # 4096^3: 5 rounds, then 264 tiles stream-K
    assert not selected(4096, 4096, 4096, G)                  # ... but 6.7 waves fill 96 % of the slots
    assert not selected(3000, 6000, 4096, G)                  # 7.4 waves: 93 %
    assert selected(2500, 2000, 2300, G)                      # 2.1 waves: 70 %
    assert not selected(1024, 1024, 4096, G)                  # 64 tiles: less than one wave
    assert not selected(4096, 4096, 1024, G)                  # short k: 64-row one-tile-per-block form
    assert plan(152, 132, 7, G) == (1, 152, 0, 0)             # r = 0: whole tiles only
    assert plan(153, 128, 0, G)[:2] == (2, 153) and plan(153, 128, 1, G)[0] == 1   # r KT < G
    assert not selected(2432, 1000, 2100, G) and not selected(2100, 1100, 2048, G)
    # the ragged shapes the GPU parity tests run through the persistent kernel:
    # one round then stream-K, no rounds, three rounds then stream-K
    for shape, n_dp in [((2432, 2100, 2050), 1), ((2500, 2000, 2300), 1), ((2000, 2000, 4100), 0),
                        ((500, 20000, 2050), 3)]:
        assert selected(*shape, G)
        per_cta, tiles, kt = segments(*shape, G)
        assert plan(tiles, kt, 0, G)[0] == n_dp
        assert sum(roles(s, kt).count("head") for s in per_cta) > 100


def test_head_plus_tail_is_the_full_sum_on_integers():
    # A scaled-down grid runs the same schedule: 5 x 3 tiles on 4 CTAs = two
    # rounds of whole tiles, then 7 tiles cut into 4 stream-K runs.
    rng = np.random.default_rng(7)
    m, n, k, grid = 600, 260, 96, 4
    kt = k // BK
    tiles_m = -(-m // BM)
    per_cta, tiles, _ = segments(m, n, k, grid)
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
    """(tile width, tiles, KT, stream-K) the launcher picks: 256 x BN tiles when
    k >= 3072, else 128 x BN.  Stream-K (always with BN = 256) when the plan
    has a region and whole tiles would fill less than 3/4 of the occupied CTA
    slots; otherwise TF32 takes BN = 224 when that fills them better by more
    than 2 %."""
    bm = 256 if k >= 3072 else 128
    kt = -(-k // (32 if mode == "tf32" else 64))

    def fill(bn):
        tiles = -(-m // bm) * -(-n // bn)
        return m * n / (-(-tiles // G) * G * bm * bn), tiles

    tiles = fill(256)[1]
    waves = -(-tiles // G)
    r = tiles % G
    if tiles >= G and r > 0 and r * kt >= G and 4 * tiles < 3 * waves * G:
        return 256, tiles, kt, True
    bn = 224 if mode == "tf32" and fill(224)[0] > 1.02 * fill(256)[0] else 256
    return bn, fill(bn)[1], kt, False


def test_umma_choices_on_the_benchmarked_shapes():
    assert umma_choice(4096, 4096, 4096, "tf32") == (224, 304, 128, False)   # 2 full waves
    assert umma_choice(8192, 8192, 8192, "bf16")[::3] == (256, False)        # 1024 tiles: 96 % filled
    assert umma_choice(4097, 3001, 1023, "tf32")[0] == 256


@pytest.mark.parametrize("mode", ["tf32", "bf16"])
def test_umma_stream_k_shapes(mode):
    G = 152
    # the GPU parity shapes for the split path: wide with no whole-tile round,
    # narrow, wide with a round
    for shape in [(3300, 3000, 3100), (2000, 2600, 1000), (2600, 4000, 4100)]:
        bn, tiles, kt, sk = umma_choice(*shape, mode)
        assert sk, shape
        per_cta = []
        for b in range(G):
            n_dp, t_sk0, v, v1 = plan(tiles, kt, b, G)
            segs = [(b + j * G, 0, kt) for j in range(n_dp)]
            while v < v1:
                q, ka = divmod(v, kt)
                kz = min(kt, ka + (v1 - v))
                segs.append((t_sk0 + q, ka, kz))
                v += kz - ka
            per_cta.append(segs)
        assert sum(roles(s, kt).count("head") for s in per_cta) > 20
    assert not umma_choice(1024, 1024, 1024, mode)[3]   # fewer tiles than SMs
