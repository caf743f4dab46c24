"""Occupancy arithmetic of the pages, on the CPU.

coffeejoa.com "CUDA.3 Writing CUDA SIMT Kernels", "Kernel Launch and
Occupancy": blocks resident per SM are limited by threads per SM, blocks per
SM, shared memory per SM and registers per SM; occupancy is resident warps over
the SM's maximum.  The page's three worked cases (2048 threads and 32 blocks
per SM): 768-thread blocks -> 2 blocks, 75 %; 32-thread blocks -> 32 blocks,
50 %; 100 KB of shared memory per block against about 233 KB per SM -> 2 blocks.
hecess.blogspot.com "[Multi-Core & GPU Programming] CUDA - Matrix
Multiplication", "Tile Size 결정": on a 2048-thread, 96 KB SM, 8x8, 16x16 and
32x32 tiles all fill the SM's threads and all use 16 KB of shared memory.

The same model, fed the launch configurations of libtgemm's kernels and
GB300's limits, must give the per-SM block counts the design relies on (and
that ncu reported as its block limits).
"""
import pytest


def blocks_per_sm(threads, smem_per_block=0, regs_per_thread=0, *, max_threads=2048, max_blocks=32,
                  smem_per_sm=None, regs_per_sm=65536, reserved_smem_per_block=0):
    limits = [max_threads // threads, max_blocks]
    if smem_per_block and smem_per_sm:
        limits.append(smem_per_sm // (smem_per_block + reserved_smem_per_block))
    if regs_per_thread:
        limits.append(regs_per_sm // (regs_per_thread * threads))
    return min(limits)


def occupancy(threads, blocks, max_threads=2048):
    return threads * blocks / max_threads


def test_case_1_thread_limited():
    b = blocks_per_sm(768)
    assert b == 2 and occupancy(768, b) == 0.75


def test_case_2_block_limited():
    b = blocks_per_sm(32)
    assert b == 32 and occupancy(32, b) == 0.5


def test_case_3_shared_memory_limited():
    assert blocks_per_sm(256, smem_per_block=100 * 1024, smem_per_sm=233 * 1024) == 2


@pytest.mark.parametrize("tile", [8, 16, 32])
def test_tile_sizes_all_use_16_kb_per_sm(tile):
    threads = tile * tile
    smem = 2 * tile * tile * 4                    # subTileM and subTileN, fp32
    b = blocks_per_sm(threads, smem, smem_per_sm=96 * 1024)
    assert b * threads == 2048                    # all thread slots used
    assert b * smem == 16 * 1024                  # but only 16 KB of the 96 KB


# GB300: 2048 threads, 32 blocks, 228 KiB of shared memory (1 KiB reserved per
# block) and 64 Ki registers per SM.
GB300 = dict(max_threads=2048, max_blocks=32, smem_per_sm=228 * 1024, regs_per_sm=65536,
             reserved_smem_per_block=1024)


@pytest.mark.parametrize("name,threads,smem,regs,expect", [
    ("ffma_f32_ws_kernel", 384, 132224, 168, 1),      # 168 at launch: 24 (producers) / 240 (consumers)
    ("ffma_f32_reduce_kernel", 256, 0, 112, 2),      # 106 registers allocate as 112
    ("umma_kernel, 4 epilogue warps", 192, 230512, 128, 1),   # 192 KiB ring + 32 KiB staging
    ("umma_kernel, 8 epilogue warps", 320, 230512, 128, 1),   # 75-127 registers
    ("umma_skinny_kernel<16>", 128, 74840, 32, 3),
    ("umma_pieces_reduce_kernel", 256, 0, 40, 6),     # register-limited: 65536 / (256 x 40)
    ("transpose_tma_kernel", 256, 99360, 40, 2),
])
def test_libtgemm_kernels(name, threads, smem, regs, expect):
    assert blocks_per_sm(threads, smem, regs, **GB300) == expect, name
