"""Shared-memory bank model and the kernels' access patterns, on the CPU.

The model is the one the pages give (note.jhbae.stream "Lec 29 · GPU
Architecture (2)", shared-memory banks; coffeejoa.com "CUDA.3 Writing CUDA
SIMT Kernels", "Shared Memory Bank Conflict"): 32 banks of 4 bytes,
consecutive words in consecutive banks, one word per bank per cycle; threads
that read the same word share it (broadcast); threads that read different
words of one bank are served one after another (an N-way conflict costs N
passes).  A 16-byte access covers four consecutive banks.  The number of
passes ("wavefronts") of a warp-wide access is the largest number of
distinct words any bank must deliver.

The FFMA kernel's addressing is restated here from its source and checked to
need one pass per instruction, i.e. to have no bank conflict (the hardware's
own count for a 128-bit load, ncu's wavefronts, is at least 2 -- 2 for the A
reads, 4 for the B reads on GB300 -- and bank conflicts would add to it); the
TMA 64-byte swizzle it relies on is
checked against the kernel's own chunk formula.  So are the TMA transpose's
reads of a 128-byte-swizzled input tile and its writes of the output tile, and
the tensor-core epilogue's staging tile.
"""
import os
import re

import pytest

CSRC = os.path.join(os.path.dirname(os.path.abspath(__file__)), "..", "dense_tiled_matrix_gb300", "csrc")

BANKS = 32


def wavefronts(addresses, width=4):
    """Passes needed for one warp access: ``addresses`` are byte addresses, one per thread."""
    words_per_bank = {}
    for a in addresses:
        for w in range(a // 4, (a + width) // 4):
            words_per_bank.setdefault(w % BANKS, set()).add(w)
    return max(len(v) for v in words_per_bank.values())


def test_quiz_word_1_and_word_33_conflict():
    # Thread 0 reads word 1, thread 1 reads word 33: both in bank 1 -> 2-way conflict.
    assert wavefronts([1 * 4, 33 * 4]) == 2


def test_stride_one_and_broadcast_are_conflict_free():
    assert wavefronts([4 * t for t in range(32)]) == 1
    assert wavefronts([4 * 7] * 32) == 1
    # bytes of the same word do not conflict either
    assert wavefronts([4 * 3 + (t % 4) for t in range(32)]) == 1


def test_transpose_tile_column_read_without_and_with_padding():
    # tile[32][32]: a warp reading one column hits one bank 32 times (31 replays).
    col = 5
    assert wavefronts([(r * 32 + col) * 4 for r in range(32)]) == 32
    # tile[32][33]: the extra word shifts each row by one bank -> conflict-free.
    assert wavefronts([(r * 33 + col) * 4 for r in range(32)]) == 1
    # the row read stays conflict-free with the padding
    assert wavefronts([(7 * 33 + c) * 4 for c in range(32)]) == 1


def swizzle64(offset):
    """TMA 64-byte swizzle: bits [4,5] of the byte offset XOR bits [7,8]."""
    return offset ^ (((offset >> 7) & 3) << 4)


# ---- FFMA kernel (csrc/ffma_f32.cu): 128x16 fp32 A tile, 16x128 fp32 B tile ----
BK, BN = 16, 128


def ffma_lane(warp, lane):
    wm, wn = warp >> 1, warp & 1
    tm, tn = lane >> 3, lane & 7
    return wm, wn, tm, tn


def ffma_a_offset(warp, lane, i, kc):
    """Byte offset in the A stage read by (warp, lane) for its row i and 16-byte chunk kc."""
    wm, wn, tm, tn = ffma_lane(warp, lane)
    r = 32 * wm + tm + 4 * i
    chunk = kc ^ ((tm >> 1) ^ ((i & 1) << 1))
    return (r * BK + chunk * 4) * 4


def ffma_b_offset(warp, lane, k, half):
    wm, wn, tm, tn = ffma_lane(warp, lane)
    return (k * BN + 64 * wn + 4 * tn + 32 * half) * 4


def test_ffma_a_chunk_formula_is_the_tma_swizzle():
    for warp in range(8):
        for lane in range(32):
            wm, wn, tm, tn = ffma_lane(warp, lane)
            for i in range(8):
                r = 32 * wm + tm + 4 * i
                for kc in range(4):
                    logical = r * 64 + kc * 16
                    assert ffma_a_offset(warp, lane, i, kc) == swizzle64(logical)


@pytest.mark.parametrize("warp", range(8))
def test_ffma_a_reads_take_one_pass(warp):
    for i in range(8):
        for kc in range(4):
            addrs = [ffma_a_offset(warp, lane, i, kc) for lane in range(32)]
            assert wavefronts(addrs, width=16) == 1, (warp, i, kc)


def test_ffma_a_reads_would_conflict_without_the_swizzle():
    # Same rows, unswizzled layout: rows 4 apart share bank groups.
    worst = 0
    for i in range(8):
        for kc in range(4):
            addrs = []
            for lane in range(32):
                wm, wn, tm, tn = ffma_lane(0, lane)
                r = 32 * wm + tm + 4 * i
                addrs.append(r * 64 + kc * 16)
            worst = max(worst, wavefronts(addrs, width=16))
    assert worst > 1


@pytest.mark.parametrize("warp", range(8))
def test_ffma_b_reads_take_one_pass(warp):
    for k in range(BK):
        for half in range(2):
            addrs = [ffma_b_offset(warp, lane, k, half) for lane in range(32)]
            assert wavefronts(addrs, width=16) == 1, (warp, k, half)


@pytest.mark.parametrize("warp_rows", [4])
def test_ffma_thread_tiles_cover_the_cta_tile_once(warp_rows):
    # warp_rows consumer warps stacked along M, two across N: a (32 warp_rows) x 128 tile
    seen = set()
    for warp in range(2 * warp_rows):
        for lane in range(32):
            wm, wn, tm, tn = ffma_lane(warp, lane)
            for i in range(8):
                for h in range(2):
                    for j in range(4):
                        cell = (32 * wm + tm + 4 * i, 64 * wn + 4 * tn + 32 * h + j)
                        assert cell not in seen
                        seen.add(cell)
    assert seen == {(r, c) for r in range(32 * warp_rows) for c in range(128)}


# ---- TMA transpose (csrc/transpose.cu): 128 x 32 fp32 input tile, 128-byte swizzle ----
def swizzle128(offset):
    """TMA 128-byte swizzle: bits [4,6] of the byte offset XOR bits [7,9]."""
    return offset ^ (((offset >> 7) & 7) << 4)


def transpose_read(warp, lane, q):
    u = warp * 4 + q
    rb, j = u >> 3, u & 7
    r = rb * 32 + lane
    return r * 128 + ((j ^ (r & 7)) << 4), (r, j)


def test_transpose_read_address_is_the_tma_swizzle():
    for warp in range(8):
        for lane in range(32):
            for q in range(4):
                addr, (r, j) = transpose_read(warp, lane, q)
                assert addr == swizzle128(r * 128 + j * 16)


@pytest.mark.parametrize("warp", range(8))
def test_transpose_reads_one_pass_per_quarter_warp(warp):
    # A 128-bit access is served a quarter-warp at a time: each quarter must
    # touch 8 distinct 16-byte bank groups.
    for q in range(4):
        for quarter in range(4):
            addrs = [transpose_read(warp, lane, q)[0] for lane in range(8 * quarter, 8 * quarter + 8)]
            assert wavefronts(addrs, width=16) == 1, (warp, q, quarter)


def test_transpose_reads_would_conflict_without_the_swizzle():
    addrs = [(rb * 32 + lane) * 128 + 3 * 16 for rb in [0] for lane in range(8)]
    assert wavefronts(addrs, width=16) == 8


@pytest.mark.parametrize("warp", range(8))
def test_transpose_writes_one_pass(warp):
    # Output tile [32][128] floats, unswizzled: lane l writes column 32 rb + l
    # of output row 4 j + e.
    for q in range(4):
        u = warp * 4 + q
        rb, j = u >> 3, u & 7
        for e in range(4):
            addrs = [((4 * j + e) * 128 + rb * 32 + lane) * 4 for lane in range(32)]
            assert wavefronts(addrs) == 1


def test_transpose_strips_cover_the_tile_once():
    seen = set()
    for warp in range(8):
        for lane in range(32):
            for q in range(4):
                _, (r, j) = transpose_read(warp, lane, q)
                for e in range(4):
                    assert (r, 4 * j + e) not in seen
                    seen.add((r, 4 * j + e))
    assert seen == {(r, c) for r in range(128) for c in range(32)}


# ---- tensor-core epilogue (csrc/umma.cu): per-warp 32 x 32 fp32 staging tile ----
# Lane l holds row l of a 32 x 32 block (one tcgen05.ld).  The tile is a TMA
# box with 128-byte swizzle: 16-byte chunk q of row i at chunk q ^ (i % 8)
# (byte 128 i + 16 (q ^ (i % 8))).  A TMA store reads it where TMA can
# describe C; otherwise the warp reads each row back, lane l taking word l.


def epi_swizzled(row, chunk, word=0):
    return row * 128 + ((chunk ^ (row & 7)) << 4) + 4 * word


def test_epilogue_layout_matches_the_kernel():
    src = open(os.path.join(CSRC, "umma.cu")).read()
    assert "tile_buf + lane * 32 + ((q ^ (lane & 7)) << 2)" in src           # TMA path
    assert "epi + lane * 32 + ((q ^ (lane & 7)) << 2)" in src                # read-back path, same layout
    assert "epi[rr * 32 + ((q ^ (rr & 7)) << 2) + w]" in src
    assert "CU_TENSOR_MAP_SWIZZLE_128B" in src and "tma_store_2d(&tmC, tile_buf, col0, row0)" in src


def test_swizzled_tile_is_the_tma_128_byte_swizzle():
    # the TMA swizzle XORs bits [4, 6] of the byte offset with bits [7, 9]
    for row in range(32):
        for q in range(8):
            logical = row * 128 + q * 16
            assert epi_swizzled(row, q) == logical ^ (((logical >> 7) & 7) << 4)


def test_swizzled_tile_writes_one_pass_per_quarter_warp():
    # float4 store of chunk q by every lane: lane l writes row l
    for q in range(8):
        for quarter in range(4):
            addrs = [epi_swizzled(l, q) for l in range(8 * quarter, 8 * quarter + 8)]
            assert wavefronts(addrs, width=16) == 1, (q, quarter)


def test_swizzled_tile_row_reads_one_pass():
    # read-back: the warp reads row rr, lane l takes word l (chunk l / 4, word l % 4)
    for rr in range(32):
        addrs = [epi_swizzled(rr, l >> 2, l & 3) for l in range(32)]
        assert wavefronts(addrs) == 1, rr
        assert sorted(addrs) == [rr * 128 + 4 * w for w in range(32)]   # exactly the row's 32 words


def test_epilogue_tile_would_conflict_without_the_swizzle():
    plain = lambda row, chunk: row * 128 + (chunk << 4)
    # the row-wise writes of one chunk by 8 rows land in one bank group: 8 passes
    assert wavefronts([plain(l, 3) for l in range(8)], width=16) == 8


