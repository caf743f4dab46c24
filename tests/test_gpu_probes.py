"""The calibration kernels (include/tgemm_probes.h) on the GPU.

Each read-stream probe must read every byte of the buffer exactly once: its
checksum (the 32-bit words added as unsigned integers, modulo 2^64) must
equal the one computed on the host, for buffer sizes that are and are not
multiples of the TMA probe's 32 KiB chunk and of the thread counts.  The
paired-FMA probe must do every one of its FMAs: with power-of-two operands
its total is exact and known in closed form.
"""
import numpy as np
import pytest
import torch

from dense_tiled_matrix_gb300 import probes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    probes.load()


@pytest.mark.parametrize("how", ["tma", "ldg"])
@pytest.mark.parametrize("nbytes", [16, 4096, 32768, 32768 + 48, 5 * 1024 * 1024 + 272, 96 * 1024 * 1024 + 16])
def test_probe_checksum_covers_every_word(how, nbytes):
    rng = np.random.default_rng(nbytes)
    host = rng.integers(0, 2 ** 32, size=nbytes // 4, dtype=np.uint64).astype(np.uint32)
    buf = torch.from_numpy(host.view(np.int32)).cuda()
    total = torch.zeros(1, dtype=torch.int64, device="cuda")
    probes.read_stream(buf, how, total)
    torch.cuda.synchronize()
    want = int(host.astype(np.uint64).sum(dtype=np.uint64))
    got = int(total.cpu().numpy().view(np.uint64)[0])
    assert got == want, (how, nbytes, got, want)


@pytest.mark.parametrize("warps", [1, 8, 16])
@pytest.mark.parametrize("iters", [0, 1, 7, 4096])
def test_ffma2_probe_does_every_fma(warps, iters):
    a = [2.0 ** -(i % 4) for i in range(8)]          # 1, 1/2, 1/4, 1/8, ...
    b = [2.0 ** (j % 3 - 1) for j in range(8)]       # 1/2, 1, 2, ...
    ab = torch.tensor(a + b, dtype=torch.float32, device="cuda")
    out = torch.zeros(1, dtype=torch.float64, device="cuda")
    probes.ffma2(warps, iters, ab, out)
    torch.cuda.synchronize()
    threads = torch.cuda.get_device_properties(0).multi_processor_count * 32 * warps
    assert out.item() == threads * iters * sum(a) * sum(b)
