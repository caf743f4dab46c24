"""The C ABI on the host: the library loads, exports every declared symbol, and
rejects bad arguments before touching the GPU.  No product is computed here."""
import ctypes
import os
import re

import pytest

from dense_tiled_matrix_gb300 import build as tbuild
from dense_tiled_matrix_gb300 import pages, probes, tgemm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tgemm.h")
PAGES_HEADER = os.path.join(ROOT, "include", "tgemm_pages.h")
PROBES_HEADER = os.path.join(ROOT, "include", "tgemm_probes.h")


@pytest.fixture(scope="module")
def lib():
    tbuild.build()
    return tgemm.load()


def declared_functions(header=HEADER):
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tgemm_[a-z0-9_]+)\s*\(", text)))


def test_every_header_under_include_is_checked():
    headers = sorted(f for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h"))
    assert headers == ["tgemm.h", "tgemm_pages.h", "tgemm_probes.h"]


def test_probes_library_exports_its_header_and_checks_arguments():
    tbuild.build()
    lib = probes.load()
    names = declared_functions(PROBES_HEADER)
    assert names == sorted(probes.SIGNATURES)
    fake_buf, fake_sum = 0x10000000, 0x20000000
    for name in [n for n in names if n.startswith("tgemm_probe_read_")]:
        fn = getattr(lib, name)
        assert fn(fake_buf, 17, fake_sum, None) == 1          # not a multiple of 16 bytes
        assert fn(fake_buf + 8, 32, fake_sum, None) == 1      # buffer not 16-byte aligned
        assert fn(fake_buf, 32, None, None) == 1              # no sum
        assert fn(fake_buf, -16, fake_sum, None) == 1
        assert fn(None, 0, fake_sum, None) == 0               # empty: nothing queued
    # the paired-FMA probe's argument rules (refused before any CUDA call)
    ffma2 = lib.tgemm_probe_ffma2
    assert ffma2(0, 16, fake_buf, fake_sum, None) == 1        # no warps
    assert ffma2(17, 16, fake_buf, fake_sum, None) == 1       # more than 16 warps per SM
    assert ffma2(8, -1, fake_buf, fake_sum, None) == 1
    assert ffma2(8, 1 << 40, fake_buf, fake_sum, None) == 1
    assert ffma2(8, 16, None, fake_sum, None) == 1            # no operands
    assert ffma2(8, 16, fake_buf + 2, fake_sum, None) == 1    # operands not 4-byte aligned
    assert ffma2(8, 16, fake_buf, fake_sum + 4, None) == 1    # out not 8-byte aligned


def test_pages_library_exports_its_header():
    tbuild.build()
    lib = pages.load()
    names = declared_functions(PAGES_HEADER)
    assert names == sorted(pages.SIGNATURES)
    for name in names:
        assert hasattr(lib, name)


def test_pages_argument_rules_on_host():
    tbuild.build()
    lib = pages.load()
    bad = tgemm.TGEMM_ERR_INVALID_VALUE
    assert lib.tgemm_pages_tiled_f32(4, 4, 4, 16, 4, 32, 4, 64, 4, 8, None) == bad     # tile 8
    assert lib.tgemm_pages_naive_f32(-1, 4, 4, 16, 4, 32, 4, 64, 4, None) == bad
    assert lib.tgemm_pages_naive_f32(4, 4, 8, 16, 7, 32, 4, 64, 4, None) == bad      # lda < k
    assert lib.tgemm_pages_naive_f32(0, 4, 4, None, 4, None, 4, None, 4, None) == tgemm.TGEMM_OK


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("tgemm_f32", "tgemm_tf32", "tgemm_bf16", "tgemm_status_string",
                 "tgemm_get_device_status", "tgemm_version"):
        assert must in names


def test_every_declared_symbol_is_exported_and_bound(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in tgemm.h but not exported"
        assert name in tgemm.SIGNATURES, f"{name} has no binding"
    assert set(tgemm.SIGNATURES) == set(declared_functions())


def test_status_strings_and_version(lib):
    for code in range(8):
        text = tgemm.tgemm_status_string(code)
        assert text and text != "unknown status"
    assert tgemm.tgemm_status_string(99) == "unknown status"
    assert tgemm.tgemm_version() >= 100
    assert tgemm.tgemm_kernel_launches() == 0


def _call(lib, name, m, n, k, A, lda, B, ldb, C, ldc):
    return getattr(lib, name)(m, n, k, A, lda, B, ldb, C, ldc, None)


FAKE_A, FAKE_B, FAKE_C = 0x10000000, 0x20000000, 0x30000000


@pytest.mark.parametrize("name", ["tgemm_f32", "tgemm_tf32", "tgemm_bf16"])
def test_argument_rules_on_host(lib, name):
    bad = tgemm.TGEMM_ERR_INVALID_VALUE
    assert _call(lib, name, -1, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4) == bad
    assert _call(lib, name, 4, 4, 1 << 31, FAKE_A, 1 << 31, FAKE_B, 4, FAKE_C, 4) == bad
    assert _call(lib, name, 4, 4, 8, FAKE_A, 7, FAKE_B, 4, FAKE_C, 4) == bad      # lda < k
    assert _call(lib, name, 4, 5, 8, FAKE_A, 8, FAKE_B, 4, FAKE_C, 5) == bad      # ldb < n
    assert _call(lib, name, 4, 5, 8, FAKE_A, 8, FAKE_B, 5, FAKE_C, 4) == bad      # ldc < n
    assert _call(lib, name, 4, 4, 4, None, 4, FAKE_B, 4, FAKE_C, 4) == bad        # NULL A
    assert _call(lib, name, 4, 4, 4, FAKE_A, 4, FAKE_B, 4, None, 4) == bad        # NULL C
    # C overlapping A or B
    assert _call(lib, name, 4, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_A + 8, 4) == bad
    assert _call(lib, name, 4, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_B - 16, 4) == bad
    # misaligned C
    assert _call(lib, name, 4, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C + 2, 4) == bad
    assert "lda" in tgemm.tgemm_last_error() or tgemm.tgemm_last_error()


@pytest.mark.parametrize("name", ["tgemm_f32", "tgemm_tf32", "tgemm_bf16"])
def test_empty_output_is_a_noop(lib, name):
    assert _call(lib, name, 0, 4, 4, None, 4, None, 4, None, 4) == tgemm.TGEMM_OK
    assert _call(lib, name, 4, 0, 4, None, 4, None, 1, None, 1) == tgemm.TGEMM_OK


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(tgemm, "_lib", None)
    with pytest.raises(ImportError):
        tgemm.load(str(tmp_path / "nope.so"))
