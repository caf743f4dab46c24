"""The debug build (libtgemm_debug.so: the same sources compiled with
TGEMM_DEBUG) on the GPU.

It carries device-side consistency checks in place of a memory checker: every
pipeline wait checks that its stage holds the fill it expects (no older fill,
no refill before the release) and, where plain threads release a stage, that
every consumer released every earlier fill; shared-memory and tensor-memory
indexes and the split-tile hand-over are checked against their buffers.  A
failed check records TGEMM_ERR_INTERNAL with its file and line in the device
status word and skips the guarded access; nothing traps.  These are the races
the pages' two barriers per phase guard against (hecess.blogspot.com
"[Multi-Core & GPU Programming] CUDA - Matrix Multiplication", "Tiled Matrix
Multiplication Kernel", the two __syncthreads: no thread reads a tile before
it is loaded, none overwrites a tile still in use).

Every kernel path runs here on small and edge cases, ragged tiles, split tiles
(fp32 k-pieces, tensor-core stream-K and split-K pieces, skinny split
tiles) and re-pitched
operands; each output must match the oracle (exactly on integer inputs) and
the status word must stay clear.  The reporting path itself is exercised with
tgemm_selftest_debug_check, which records a failed check without any other
effect.
"""
import numpy as np
import pytest
import torch

import oracle
from dense_tiled_matrix_gb300 import inputs, tgemm
import parity

pytestmark = pytest.mark.gpu

ENTRY = {"f32": tgemm.tgemm_f32, "tf32": tgemm.tgemm_tf32, "bf16": tgemm.tgemm_bf16}


@pytest.fixture(scope="module")
def dbg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    lib = tgemm.open_library(tgemm.DEBUG_LIB_PATH)
    assert lib.tgemm_debug_build() == 1
    assert tgemm.load().tgemm_debug_build() == 0
    yield lib
    assert lib.tgemm_get_device_status(None) == tgemm.TGEMM_OK, lib.tgemm_last_error().decode()


def _check(dbg, mode, case, what):
    A_np, B_np = parity.inputs_for(mode, case)
    A, B = parity.to_device(A_np), parity.to_device(B_np)
    C = ENTRY[mode](A, B, lib=dbg)
    status = dbg.tgemm_get_device_status(torch.cuda.current_stream().cuda_stream)
    assert status == tgemm.TGEMM_OK, f"{what}: {dbg.tgemm_last_error().decode()}"
    P, D = oracle.gemm(A_np, B_np)
    parity.check(mode, C.cpu().numpy(), P, D, case.exact, what)


CASES = [
    # name, modes, (m, n, k) or a named workload
    ("worked_4x4", ["f32", "tf32", "bf16"]),
    ("int64", ["f32", "tf32", "bf16"]),
    ("u128", ["f32", "tf32", "bf16"]),
    ("int1024", ["f32", "tf32", "bf16"]),
    ((127, 129, 33), ["f32", "tf32", "bf16"]),
    ((129, 257, 17), ["f32", "tf32", "bf16"]),
    ((1000, 64, 65), ["f32", "tf32", "bf16"]),
    ((257, 511, 257), ["f32", "tf32", "bf16"]),
    ((300, 520, 3100), ["f32", "tf32", "bf16"]),        # 256 x 256 tensor-core tiles as split-K pieces
    ((1000, 1001, 2000), ["tf32", "bf16"]),               # 128 x 256 tiles as split-K pieces, C unaligned
    ((1000, 900, 4100), ["f32"]),                         # fp32 k-pieces + ordered reduce
    ((3300, 3000, 3100), ["tf32", "bf16"]),               # tensor-core stream-K
    ((2000, 2600, 1000), ["tf32", "bf16"]),               # stream-K with 128 x 256 tiles
    ((16, 8192, 8192), ["bf16"]),                         # skinny, split tiles
    ((33, 129, 70), ["bf16"]),
    ((64, 4096, 8192), ["bf16"]),
    ((3, 20000, 4160), ["bf16"]),
    ((4097, 3001, 1023), ["f32", "tf32", "bf16"]),       # every operand re-pitched
    ((2000, 4800, 999), ["bf16"]),                        # multicast CTA pairs
]


@pytest.mark.parametrize("spec, modes", CASES, ids=lambda v: v if isinstance(v, str) else "x".join(map(str, v))
                         if isinstance(v, tuple) else "")
def test_debug_build_matches_oracle_with_no_failed_check(dbg, spec, modes):
    for mode in modes:
        if isinstance(spec, str):
            case = inputs.make(spec)
            _check(dbg, mode, case, f"debug {mode} {spec}")
        else:
            m, n, k = spec
            for kind in ("int", "uniform"):
                case = inputs.random_case(15000 + m + 3 * n + 7 * k, m, n, k, kind=kind)
                _check(dbg, mode, case, f"debug {mode} {kind} {spec}")


def test_a_failed_check_is_reported_with_its_place(dbg):
    stream = torch.cuda.current_stream().cuda_stream
    assert dbg.tgemm_selftest_debug_check(stream) == tgemm.TGEMM_OK
    assert dbg.tgemm_get_device_status(stream) == tgemm.TGEMM_ERR_INTERNAL
    assert "selftest.cu" in dbg.tgemm_last_error().decode()
    assert dbg.tgemm_get_device_status(stream) == tgemm.TGEMM_OK      # read and cleared
    # the context is still usable
    _check(dbg, "f32", inputs.make("int64"), "debug f32 int64 after the reported check")
