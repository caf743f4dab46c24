"""The tensor-core launcher's tile choices (csrc/umma.cu), restated for the tests.

Tile height: 256-row ("wide") tiles when k >= 3072; for 1024 <= k < 3072
where the wide grid needs no stream-K and fills its rounds of CTAs at least
as well as the 128-row grid (a 128-row grid with stream-K counts as full);
otherwise 128-row tiles.  Stream-K: the persistent plan has a region (T = qG
+ r tiles, q >= 1, r > 0, r * KT >= G) and whole tiles would fill less than
3/4 of their CTA slots.  Split-K pieces: fewer tiles than CTAs (see pieces).
"""


def k_phases(k, mode):
    """Phases of 128 bytes of k."""
    return -(-k // (32 if mode == "tf32" else 64))


def tiles_of(m, n, bm, bn=256):
    return -(-m // bm) * -(-n // bn)


def stream_k(tiles, kt, G=152):
    r = tiles % G
    waves = -(-tiles // G)
    return tiles >= G and r > 0 and r * kt >= G and 4 * tiles < 3 * waves * G


def slot_fill(m, n, bm, bn=256, G=152):
    """Filled fraction of the CTA slots the whole-tile grid occupies."""
    t = tiles_of(m, n, bm, bn)
    return m * n / (-(-t // G) * G * bm * bn)


def tile_rows(m, n, k, mode, G=152):
    """256 or 128: the height of the tensor-core tiles the launcher picks."""
    if k >= 3072:
        return 256
    if k < 1024:
        return 128
    kt = k_phases(k, mode)
    if stream_k(tiles_of(m, n, 256), kt, G):
        return 128
    narrow = 1.0 if stream_k(tiles_of(m, n, 128), kt, G) else slot_fill(m, n, 128, G=G)
    return 256 if slot_fill(m, n, 256, G=G) >= narrow else 128


def pieces(m, n, k, mode, G=152):
    """Split-K pieces per tile (0: none): where the whole tiles (of the height
    tile_rows picks, 256 wide) fill less than one round of CTAs, each tile is
    cut along k into as many pieces as fit in one round, each at least 8
    k-phases long; at least 2."""
    tiles = tiles_of(m, n, tile_rows(m, n, k, mode, G))
    if tiles >= G:
        return 0
    p = min(G // tiles, k_phases(k, mode) // 8)
    return p if p >= 2 else 0


def tile_cols(m, n, k, mode, G=152):
    """256, or 224 for TF32 where the whole tiles take neither stream-K nor
    pieces and 224-wide ones fill the occupied CTA slots better by more than 2 %."""
    if mode != "tf32":
        return 256
    bm = tile_rows(m, n, k, mode, G)
    if stream_k(tiles_of(m, n, bm), k_phases(k, mode), G) or pieces(m, n, k, mode, G):
        return 256
    return 224 if slot_fill(m, n, bm, 224, G) > 1.02 * slot_fill(m, n, bm, 256, G) else 256


def pairs(m, n, k, G=152):
    """bf16 128 x 256 whole tiles as multicast CTA pairs: no stream-K, no pieces,
    an even number of tile rows and at least two rounds of tiles."""
    if tile_rows(m, n, k, "bf16", G) != 128:
        return False
    tiles = tiles_of(m, n, 128)
    if stream_k(tiles, k_phases(k, "bf16"), G) or pieces(m, n, k, "bf16", G):
        return False
    return (-(-m // 128)) % 2 == 0 and tiles >= 2 * G


def plan(m, n, k, mode, G=152, workspace=True):
    """(tile rows, tile columns, stream-K, pieces, pairs) as tgemm_plan reports
    them; bf16 with m <= 64 (the cluster split-K kernel) is all zero.  Without
    workspace neither stream-K nor pieces is taken."""
    if mode == "bf16" and m <= 64:
        return (0, 0, False, 0, False)
    bm, bn = tile_rows(m, n, k, mode, G), tile_cols(m, n, k, mode, G)
    if bn == 224:
        return (bm, 224, False, 0, False)
    sk = workspace and stream_k(tiles_of(m, n, bm), k_phases(k, mode), G)
    pc = pieces(m, n, k, mode, G) if workspace and not sk else 0
    pr = mode == "bf16" and not sk and not pc and bm == 128 and (-(-m // 128)) % 2 == 0 \
        and tiles_of(m, n, 128) >= 2 * G
    return (bm, bn, sk, pc, pr)
