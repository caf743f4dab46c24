"""bench.py's host-side arithmetic, on the CPU: the roofline object of each path
and the parsing of the nvidia-smi clock log (no GPU, no subprocess)."""
import os
from collections import namedtuple

import pytest

import bench

Case = namedtuple("Case", "m n k")
PEAKS = {"hbm_gbs": 6792.0, "bf16_tflops": 1904.1}


def test_skinny_bf16_is_hbm_bound_on_algorithmic_bytes():
    c = Case(16, 8192, 8192)
    r = bench.roofline_for("bf16", c, 28.0e-6, PEAKS, "measured")
    nbytes = 2 * (16 * 8192 + 8192 * 8192) + 4 * 16 * 8192   # A and B read once (bf16), C written once (fp32)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["algorithmic_bytes"] == nbytes
    assert r["achieved"] == pytest.approx(nbytes / 28.0e-6 / 1e9, abs=0.05)
    assert r["frac"] == pytest.approx(r["achieved"] / 6792.0, abs=1e-4)


@pytest.mark.parametrize("entry, bound, peak, nominal", [
    ("f32", "alu", 148 * 128 * 2 * 1980e6 / 1e12, None),
    ("pages_naive", "alu", 148 * 128 * 2 * 1980e6 / 1e12, None),
    ("bf16", "tensor", 1904.1, 2250.0),
    ("tf32", "tensor", 1904.1 * 1100.0 / 2250.0, 1100.0),
])
def test_compute_bound_paths_use_their_own_peak(entry, bound, peak, nominal):
    c = Case(4096, 4096, 4096)
    fp32 = bench.fp32_peak(148, 1980.0)      # SM count and clock as read at run time
    r = bench.roofline_for(entry, c, 2.0e-3, PEAKS, "measured", fp32)
    flops = 2.0 * 4096 ** 3
    assert r["bound"] == bound and r["unit"] == "TFLOP/s" and r["algorithmic_flops"] == int(flops)
    assert r["peak"] == pytest.approx(peak, abs=0.01)
    assert r["achieved"] == pytest.approx(flops / 2.0e-3 / 1e12, abs=0.01)
    assert r["frac"] == pytest.approx(flops / 2.0e-3 / 1e12 / peak, abs=1e-4)
    if nominal is None:
        assert "148 SMs" in r["peak_source"] and "1980 MHz" in r["peak_source"]
        assert "frac_of_nominal" not in r
    else:
        assert r["nominal_peak"] == nominal
        assert r["frac_of_nominal"] == pytest.approx(flops / 2.0e-3 / 1e12 / nominal, abs=1e-4)


def test_fp32_peak_derivation():
    tf, how = bench.fp32_peak(152, 2070.0)
    assert tf == pytest.approx(152 * 128 * 2 * 2070e6 / 1e12)
    assert how.startswith("152 SMs x 128 FP32 lanes x 2 flop x 2070 MHz")


def test_traffic_table_parses_and_matches_its_sources():
    """Every row of the committed ncu traffic table parses; a row whose kernel
    sources are unchanged gives its bytes, a changed one gives None."""
    table = bench.traffic_table()
    assert {"f32_4096", "bf16_8192"} <= set(table)
    for part, row in table.items():
        assert row["source"].startswith("profiles/")
        if not row["stale"]:
            assert isinstance(row["bytes"], int) and row["bytes"] > 0, part
        else:
            assert row["bytes"] is None, part


def test_traffic_table_marks_changed_sources_stale(tmp_path):
    path = tmp_path / "t.csv"
    digest = bench.source_digest(["ffma_f32.cu"])
    path.write_text("# comment\npart,bytes_per_call,kernels,sources,sha256_16,summary\n"
                    f"a,100,k,ffma_f32.cu,{digest},profiles/x.md\n"
                    "b,200,k,ffma_f32.cu,0000000000000000,profiles/y.md\n")
    table = bench.traffic_table(str(path))
    assert table["a"] == {"bytes": 100, "source": "profiles/x.md (k)", "stale": False}
    assert table["b"]["bytes"] is None and table["b"]["stale"]


def _summary(tmp_path, lines):
    s = bench.ClockSampler(0)
    s.path = os.path.join(tmp_path, "clocks.csv")   # as if __enter__ had made it
    with open(s.path, "w") as fh:
        fh.write("\n".join(lines) + "\n")
    s.proc = object()   # as if nvidia-smi had run
    return s.summary()


def test_clock_log_median_and_no_reasons(tmp_path):
    rows = [f"0, {mhz}, 2070, 450.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active"
            for mhz in (2070, 2055, 2070, 1980, 2070)]
    out = _summary(tmp_path, rows)
    assert out["sm_mhz"] == 2070 and out["sm_max_mhz"] == 2070 and out["reasons"] == []
    assert out["samples"] == 5 and out["power_w_max"] == 450.5


def test_clock_log_reports_every_throttle_reason_seen(tmp_path):
    rows = ["0, 2070, 2070, 900.0, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 1800, 2070, 1300.0, 0x48, Not Active, Active, Not Active, Active",
            "0, 2070, 2070, 800.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "garbled line"]
    out = _summary(tmp_path, rows)
    assert out["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert out["samples"] == 3 and out["sm_mhz"] == 2070


def test_clock_log_without_samples(tmp_path):
    out = _summary(tmp_path, [""])
    assert out["reasons"] == ["no samples"] and out["sm_mhz"] is None


def test_every_bench_shape_names_a_workload_and_an_entry():
    """Each part of the step and each extra shape names a seeded workload that
    inputs.make builds (sizes as the bench docstring states them) and an entry
    point the bench knows; the two split-K extras have fewer tensor-core tiles
    than SMs."""
    from dense_tiled_matrix_gb300 import inputs
    import launch_rules
    entries = {"f32", "tf32", "bf16", "pages_naive", "pages_tiled16", "pages_tiled32"}
    sizes = {}
    for name, (wl, entry, _) in list(bench.PARTS.items()) + list(bench.EXTRAS.items()):
        assert entry in entries, name
        if wl not in sizes:
            c = inputs.make(wl)
            sizes[wl] = (c.m, c.n, c.k)
    assert sizes["bf16_8192"] == (8192, 8192, 8192) and sizes["n4096"] == (4096, 4096, 4096)
    assert sizes["skinny"] == (16, 8192, 8192) and sizes["irregular"] == (4097, 3001, 1023)
    assert sizes["long_k"] == (1024, 1024, 8192)
    for mode in ("bf16", "tf32"):
        assert launch_rules.pieces(*sizes["long_k"], mode) >= 2


def test_plan_of_each_entry():
    """bench.plan_of reports libtgemm's own plan for the shapes it times
    (host arithmetic, no GPU): FFMA split remainder at 4096^3, wide tiles at
    8192^3, TF32 224-wide tiles at 4096^3, split-K pieces at 1024 x 1024 x 8192;
    nothing for the pages' kernels."""
    from dense_tiled_matrix_gb300 import build as tbuild
    tbuild.build()
    assert bench.plan_of("f32", 4096, 4096, 4096, 152) == {"whole_tiles": 912, "split_tiles": 112, "pieces": 4}
    assert bench.plan_of("bf16", 8192, 8192, 8192, 152)["tile_rows"] == 256
    assert bench.plan_of("tf32", 4096, 4096, 4096, 152)["tile_cols"] == 224
    assert bench.plan_of("bf16", 1024, 1024, 8192, 152)["pieces"] == 9
    assert bench.plan_of("bf16", 16, 8192, 8192, 152)["tile_rows"] == 0    # the cluster split-K kernel
    assert bench.plan_of("pages_naive", 1024, 1024, 1024, 152) is None
