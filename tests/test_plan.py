"""The tensor-core tile plan: the library's own choice (tgemm_plan, host
arithmetic, no GPU) against the rules the tests restate (launch_rules.py).

The GPU parity tests pick their shapes from the restated rules (stream-K,
split-K pieces, CTA pairs, 256-row and 224-wide tiles); this checks, on the
CPU, that the library makes exactly those choices, over the tests' shapes,
the benchmarked ones and a seeded sweep around every boundary of the rules."""
import numpy as np
import pytest

import launch_rules
from dense_tiled_matrix_gb300 import build as tbuild
from dense_tiled_matrix_gb300 import tgemm


@pytest.fixture(scope="module", autouse=True)
def _lib():
    tbuild.build()
    tgemm.load()


def library_plan(m, n, k, mode, G=152, workspace=True):
    d = tgemm.tgemm_plan(mode, m, n, k, G, workspace)
    return (d["tile_rows"], d["tile_cols"], d["stream_k"], d["pieces"], d["pairs"])


NAMED = [
    (8192, 8192, 8192), (4096, 4096, 4096), (16, 8192, 8192), (4097, 3001, 1023), (1024, 1024, 1024),
    (3300, 3000, 3100), (2000, 2600, 1000), (2600, 4000, 4100), (2048, 4864, 1000), (2000, 4800, 999),
    (4096, 2432, 200), (1536, 9728, 1024), (2048, 4864, 1024), (2900, 5000, 1030), (1024, 1024, 8192),
    (65, 4096, 4096), (1000, 1001, 2000), (129, 1000, 3072), (300, 520, 3100), (256, 256, 65536),
    (4100, 8200, 16), (2048, 2048, 2048), (8192, 8192, 1024), (6144, 3072, 1024), (64, 4096, 8192),
]


@pytest.mark.parametrize("mode", ["bf16", "tf32"])
def test_library_plan_matches_the_restated_rules_on_named_shapes(mode):
    for shape in NAMED:
        for ws in (True, False):
            assert library_plan(*shape, mode, workspace=ws) == launch_rules.plan(*shape, mode, workspace=ws), \
                (shape, mode, ws)


@pytest.mark.parametrize("mode", ["bf16", "tf32"])
def test_library_plan_matches_the_restated_rules_on_a_sweep(mode):
    """Sizes near multiples of 128 / 224 / 256 and tile counts near multiples of
    the SM count, k around the thresholds (8 k-phases a piece, 1024, 3072)."""
    rng = np.random.default_rng(20)
    near = lambda base: int(max(1, base + rng.integers(-2, 3)))
    seen = set()
    for _ in range(3000):
        m = near(int(rng.choice([65, 128, 256, 640, 1024, 1536, 2048, 2432, 3072, 4096, 6144, 8192])))
        n = near(int(rng.choice([128, 224, 256, 448, 1024, 2432, 3001, 4864, 9728])))
        k = near(int(rng.choice([16, 256, 512, 1000, 1024, 2048, 3072, 4096, 65536])))
        G = int(rng.choice([152, 148, 132]))
        ours = library_plan(m, n, k, mode, G)
        assert ours == launch_rules.plan(m, n, k, mode, G), (m, n, k, mode, G)
        seen.add((ours[0], ours[1], ours[2], ours[3] > 0, ours[4]))
    # the sweep reached every kind of plan the launcher has
    kinds = {(s[0], s[1], s[2], s[3], s[4]) for s in seen}
    assert any(s[2] for s in kinds) and any(s[3] for s in kinds)
    assert any(s[0] == 256 for s in kinds) and any(s[0] == 128 for s in kinds)
    if mode == "bf16":
        assert any(s[4] for s in kinds)
    else:
        assert any(s[1] == 224 for s in kinds)


def test_plan_argument_rules():
    import ctypes
    lib = tgemm.load()
    out = (ctypes.c_int * 5)(*([7] * 5))
    bad = tgemm.TGEMM_ERR_INVALID_VALUE
    assert lib.tgemm_plan(0, 0, 4, 4, 152, 1, out) == bad
    assert lib.tgemm_plan(0, 4, 4, 1 << 31, 152, 1, out) == bad
    assert lib.tgemm_plan(0, 4, 4, 4, 0, 1, out) == bad
    assert lib.tgemm_plan(0, 4, 4, 4, 152, 1, None) == bad
    assert list(out) == [7] * 5                      # untouched on a refusal
    assert lib.tgemm_plan(0, 16, 4, 4, 152, 1, out) == tgemm.TGEMM_OK
    assert list(out) == [0] * 5                      # bf16, m <= 64: the cluster split-K kernel
    out64 = (ctypes.c_int64 * 3)(7, 7, 7)
    assert lib.tgemm_plan_f32(4, 0, 4, 152, out64) == bad
    assert lib.tgemm_plan_f32(4, 4, 4, 5000, out64) == bad
    assert lib.tgemm_plan_f32(4, 4, 4, 152, None) == bad
    assert list(out64) == [7, 7, 7]
    assert lib.tgemm_plan_f32(4, 4, 4, 152, out64) == tgemm.TGEMM_OK and list(out64) == [1, 0, 0]


def test_fp32_plan_matches_the_restated_split_rule():
    """tgemm_f32's split of a partly filled last round (tgemm_plan_f32) against
    test_stream_k_model.split_tail, on named shapes and a seeded sweep of tile
    counts around multiples of the SM count and k around the piece minimum."""
    from test_stream_k_model import split_tail

    def library(m, n, k, G):
        d = tgemm.tgemm_plan_f32(m, n, k, G)
        return None if d["pieces"] == 0 else (d["whole_tiles"], d["split_tiles"], d["pieces"])

    for shape in [(4096, 4096, 4096), (1024, 1024, 4096), (8192, 8192, 2048), (4097, 3001, 1023),
                  (8192, 8192, 512), (200, 150, 90), (256, 256, 65536), (2432, 2100, 2050), (1000, 900, 4100),
                  (500, 20000, 2050), (2000, 2000, 4100), (1024, 1024, 1024)]:
        assert library(*shape, 152) == split_tail(*shape), shape
    rng = np.random.default_rng(21)
    split = 0
    for _ in range(3000):
        m = int(rng.integers(1, 9000))
        n = int(rng.integers(1, 9000))
        k = int(rng.choice([16, 200, 255, 256, 257, 511, 1024, 4100, 70000]))
        G = int(rng.choice([152, 148, 132]))
        want = split_tail(m, n, k, G)
        assert library(m, n, k, G) == want, (m, n, k, G)
        if want is None:
            d = tgemm.tgemm_plan_f32(m, n, k, G)
            assert d["whole_tiles"] == -(-m // 128) * -(-n // 128) and d["split_tiles"] == 0
        else:
            split += 1
    assert 300 < split < 2700     # both kinds of plan were reached
