"""Row sharding of one product over several ranks (one GPU per rank).

P = M x N splits by rows with no communication: rank r of W computes the row
block rows(m, W, r) of C from the same rows of A and the whole of B, each an
independent call of the C entry point on its own GPU.  Gathering the blocks
is only needed by a caller that wants all of C on every rank; the product
itself has no collective.
"""
from __future__ import annotations


def rows(m: int, world: int, rank: int) -> tuple[int, int]:
    """Half-open row range [r0, r1) of rank ``rank``; blocks differ in size by at most one row."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    return (m * rank) // world, (m * (rank + 1)) // world


def local_product(product, A, B, world: int, rank: int):
    """This rank's block of C = A @ B computed with ``product(A_block, B)``."""
    r0, r1 = rows(A.shape[0], world, rank)
    return r0, r1, product(A[r0:r1], B)


def gather_rows(block, m: int, world: int, group=None):
    """All ranks' row blocks stacked into the full C (torch.distributed all_gather)."""
    import torch
    import torch.distributed as dist
    sizes = [rows(m, world, r)[1] - rows(m, world, r)[0] for r in range(world)]
    pad = max(sizes)
    buf = torch.zeros((pad, block.shape[1]), dtype=block.dtype, device=block.device)
    buf[: block.shape[0]] = block
    parts = [torch.empty_like(buf) for _ in range(world)]
    dist.all_gather(parts, buf, group=group)
    return torch.cat([p[:s] for p, s in zip(parts, sizes)], dim=0)
