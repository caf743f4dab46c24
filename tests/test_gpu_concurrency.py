"""Several host threads calling the library at once, each on its own stream.

The library keeps no per-call state outside the call: the error text is
thread-local, the device table is set up once under a lock, and every
workspace (re-pitched operands, the TF32 B transpose, fp32 k-pieces,
tensor-core stream-K and split-K partials) is stream-ordered memory of the
calling stream.  So concurrent calls on different streams must give the same
results as calls one at a time: here every result must equal the oracle
exactly (integer inputs) while four threads run all the workspace-using
paths at the same time.  (`tgemm_tf32_noalloc` shares one static scratch
array by design and is not called concurrently.)
"""
import threading

import numpy as np
import pytest
import torch

import oracle
from dense_tiled_matrix_gb300 import inputs, tgemm
import parity

pytestmark = pytest.mark.gpu

CASES = [
    ("f32", (1000, 900, 4100)),     # fp32 k-pieces + ordered reduce (workspace)
    ("f32", (1025, 700, 301)),      # misaligned rows: re-pitch (workspace)
    ("tf32", (300, 520, 200)),      # B transpose (workspace)
    ("bf16", (2000, 2600, 1000)),   # tensor-core stream-K (workspace)
    ("tf32", (300, 520, 3100)),     # split-K pieces + reduce (workspace)
    ("bf16", (16, 1000, 4100)),     # skinny cluster split
    ("bf16", (257, 511, 257)),      # whole tiles, ragged edges
    ("bf16", (2048, 4864, 1000)),   # multicast CTA pairs (cluster launches)
    ("bf16", (2048, 4864, 1024)),   # 256-row tiles at k < 3072 (one exact round)
]
THREADS = 4
REPEATS = 3


@pytest.fixture(scope="module")
def cases():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    out = []
    for i, (mode, (m, n, k)) in enumerate(CASES):
        case = inputs.random_case(12000 + i, m, n, k, kind="int")
        A, B = parity.inputs_for(mode, case)
        P, _ = oracle.gemm(A, B)
        out.append((mode, A, B, P.astype(np.float32)))
    return out


def test_concurrent_calls_on_separate_streams_match_the_oracle(cases):
    errors = []
    results = {}
    start = threading.Barrier(THREADS)

    def worker(t):
        try:
            torch.cuda.set_device(0)
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                dev = [(mode, parity.to_device(A), parity.to_device(B)) for mode, A, B, _ in cases]
                outs = [[torch.full((A.shape[0], B.shape[1]), float("nan"), device="cuda") for _ in range(REPEATS)]
                        for _, A, B in dev]
                stream.synchronize()
                start.wait(timeout=300)
                for r in range(REPEATS):
                    for i, (mode, A, B) in enumerate(dev):
                        parity.ENTRY[mode](A, B, outs[i][r], stream=stream)
                stream.synchronize()
                results[t] = [[o.cpu().numpy() for o in row] for row in outs]
        except Exception as exc:   # reported on the main thread
            errors.append((t, repr(exc)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(THREADS)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=600)
    assert not any(th.is_alive() for th in threads), "a worker thread did not finish"
    assert not errors, errors
    assert tgemm.tgemm_get_device_status() == tgemm.TGEMM_OK
    for t in range(THREADS):
        for i, (mode, A, B, P) in enumerate(cases):
            for r in range(REPEATS):
                C = results[t][i][r]
                assert np.array_equal(C, P), (t, mode, CASES[i][1], r, float(np.nanmax(np.abs(C - P))))
