"""Failure detection on the GPU without a fault or a hang.

A kernel whose pipeline wait never completes must give up after its time
limit, record TGEMM_ERR_TIMEOUT in the device status word and return; the
host reads the status, which is then cleared, and the context stays usable.
The wait that runs out is the product kernels' own bounded-wait helper, on a
barrier that nothing arrives at (tgemm_selftest_wait_timeout), with a 20 ms
limit.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from dense_tiled_matrix_gb300 import inputs, tgemm
import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    tgemm.load()


def test_timeout_is_reported_and_the_context_survives():
    assert tgemm.tgemm_get_device_status() == tgemm.TGEMM_OK
    t0 = time.perf_counter()
    assert tgemm.tgemm_selftest_wait_timeout(20_000_000) == tgemm.TGEMM_OK
    status = tgemm.tgemm_get_device_status()
    elapsed = time.perf_counter() - t0
    assert status == tgemm.TGEMM_ERR_TIMEOUT
    assert "timed out" in tgemm.tgemm_last_error()
    assert 0.015 < elapsed < 10.0
    # the status word was cleared by the read
    assert tgemm.tgemm_get_device_status() == tgemm.TGEMM_OK
    # and the GPU still computes correctly
    parity.full_check("f32", inputs.make("int64"))
    parity.full_check("bf16", inputs.make("int64"))
    assert tgemm.tgemm_get_device_status() == tgemm.TGEMM_OK


def test_selftest_rejects_bad_limits():
    assert tgemm.tgemm_selftest_wait_timeout(10) == tgemm.TGEMM_ERR_INVALID_VALUE
    assert tgemm.tgemm_selftest_wait_timeout(10 ** 12) == tgemm.TGEMM_ERR_INVALID_VALUE
