"""Row-sharded product over two ranks (gloo on the CPU).

Each rank computes its row block of P with the CPU oracle standing in for its
GPU's tgemm call; the blocks, gathered, must equal the unsharded oracle result
bit for bit (every row is the same fp64 sum in the same order).  Also checks
the row partition and the bench's max-over-ranks reduction.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from dense_tiled_matrix_gb300 import sharding


def test_row_partition_covers_every_row_once():
    for m in (0, 1, 5, 7, 64, 4097):
        for world in (1, 2, 3, 8):
            got = []
            for r in range(world):
                r0, r1 = sharding.rows(m, world, r)
                got.extend(range(r0, r1))
                assert r1 - r0 in (m // world, m // world + 1)
            assert got == list(range(m))
    with pytest.raises(ValueError):
        sharding.rows(4, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, result_path):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import sys
        root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
        sys.path.insert(0, root)
        import oracle
        from dense_tiled_matrix_gb300 import inputs
        case = inputs.random_case(31, 37, 23, 19, kind="normal")
        r0, r1, P_local = sharding.local_product(lambda a, b: oracle.gemm(a, b)[0], case.A, case.B, world, rank)
        C = sharding.gather_rows(torch.from_numpy(P_local), case.m, world)
        # the bench's timing reduction: max over ranks
        t = torch.tensor([float(rank + 1)], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        if rank == 0:
            np.save(result_path, C.numpy())
            assert t.item() == float(world)
    finally:
        dist.destroy_process_group()


def test_two_ranks_row_sharded_product_equals_unsharded(tmp_path):
    import oracle
    from dense_tiled_matrix_gb300 import inputs
    out = str(tmp_path / "c.npy")
    mp.spawn(_worker, args=(2, _free_port(), out), nprocs=2, join=True)
    case = inputs.random_case(31, 37, 23, 19, kind="normal")
    P, _ = oracle.gemm(case.A, case.B)
    assert np.array_equal(np.load(out), P)
