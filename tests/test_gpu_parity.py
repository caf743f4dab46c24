"""GPU parity: every entry point against the CPU oracle, through the C ABI.

Small and medium cases are compared element by element over the whole
output; the full-size workloads (4096^3 fp32, 8192^3 bf16) on sampled rows and
entries that the oracle evaluates one by one.  Integer-valued inputs must match
exactly; other inputs within the bounds stated in ``parity.py``.
"""
import numpy as np
import pytest
import torch

import oracle
from dense_tiled_matrix_gb300 import inputs, tgemm
import parity
import launch_rules

pytestmark = pytest.mark.gpu

MODES = ["f32", "tf32", "bf16"]


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    tgemm.load()
    yield
    assert tgemm.tgemm_get_device_status() == tgemm.TGEMM_OK


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("name", ["worked_4x4", "int64", "u128", "int1024"])
def test_named_small_cases(mode, name):
    parity.full_check(mode, inputs.make(name))


EDGE_SHAPES = [
    (1, 1, 1), (1, 7, 3), (5, 1, 9), (2, 3, 300), (127, 129, 33), (128, 128, 16), (128, 256, 64),
    (129, 257, 17), (255, 300, 31), (300, 200, 1), (513, 300, 100), (64, 1000, 129),
    (1000, 64, 65), (257, 511, 257), (130, 260, 520),
]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("shape", EDGE_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_edge_tiles(mode, shape):
    m, n, k = shape
    parity.full_check(mode, inputs.random_case(2000 + m + 7 * n + 13 * k, m, n, k, kind="int"),
                      f"{mode} int {shape}")
    parity.full_check(mode, inputs.random_case(3000 + m + 7 * n + 13 * k, m, n, k, kind="uniform"),
                      f"{mode} uniform {shape}")


# k >= 3072 always takes the 256 x 256 tensor-core tiles; ragged m, n and k there
# too (these few tiles run as split-K pieces).
WIDE_SHAPES = [(300, 520, 3100), (257, 300, 4097), (129, 1000, 3072)]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("shape", WIDE_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_long_k_tiles(mode, shape):
    m, n, k = shape
    parity.full_check(mode, inputs.random_case(5000 + m + n + k, m, n, k, kind="int"), f"{mode} int {shape}")
    parity.full_check(mode, inputs.random_case(6000 + m + n + k, m, n, k, kind="uniform"), f"{mode} uniform {shape}")


# 1024 <= k < 3072 where the 256-row tiles fill their rounds of CTAs at least
# as well as the 128-row ones and need no stream-K: they take the 256 x 256
# tiles too (one exact round of them; ragged m, n and k).
MID_K_WIDE_SHAPES = [(2048, 4864, 1024), (2900, 5000, 1030)]


@pytest.mark.parametrize("mode", ["tf32", "bf16"])
@pytest.mark.parametrize("shape", MID_K_WIDE_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_mid_k_wide_tiles(mode, shape):
    m, n, k = shape
    assert launch_rules.tile_rows(m, n, k, mode) == 256
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert tgemm.tgemm_plan(mode, m, n, k, sm)["tile_rows"] == 256
    parity.full_check(mode, inputs.random_case(5100 + m + n + k, m, n, k, kind="int"), f"{mode} int {shape}")
    parity.full_check(mode, inputs.random_case(6100 + m + n + k, m, n, k, kind="uniform"), f"{mode} uniform {shape}")


@pytest.mark.parametrize("mode", MODES)
def test_irregular_4097x3001x1023(mode):
    # lda = 1023 and ldb = ldc = 3001: no row pitch is a multiple of 16 bytes.
    parity.full_check(mode, inputs.make("irregular"))


# The fp32 split remainder (k >= 2048 and a partly empty last wave): the
# one-tile grid covers the full rounds, the tiles left are cut along k into
# pieces whose partial sums a reduce kernel adds in part order.  Full rounds
# then 19 tiles in 8 pieces; no full round (64 tiles in 7 pieces); 4 rounds
# then 20 tiles in 7; 1 round then 104 tiles in 7.  Ragged in m, n and k,
# checked over the whole output.
SPLIT_SHAPES = [(2432, 2100, 2050), (1000, 900, 4100), (500, 20000, 2050), (2000, 2000, 4100)]


@pytest.mark.parametrize("shape", SPLIT_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_fp32_split_remainder(shape):
    m, n, k = shape
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert tgemm.tgemm_plan_f32(m, n, k, sm)["pieces"] >= 2   # this device splits the last round
    parity.full_check("f32", inputs.random_case(7000 + m + n + k, m, n, k, kind="int"), f"f32 int {shape}")
    case = inputs.random_case(8000 + m + n + k, m, n, k, kind="uniform")
    parity.full_check("f32", case, f"f32 uniform {shape}")
    A, B = parity.to_device(case.A), parity.to_device(case.B)
    assert torch.equal(parity.ENTRY["f32"](A, B), parity.ENTRY["f32"](A, B))


# Tensor-core shapes whose last partial wave of tiles is split along k between
# two CTAs (stream-K): wide 256 x 256 tiles with no whole-tile round, narrow
# 128 x 256 tiles, wide tiles after one round.  Ragged, whole output checked.
UMMA_SK_SHAPES = [(3300, 3000, 3100), (2000, 2600, 1000), (2600, 4000, 4100)]


@pytest.mark.parametrize("mode", ["tf32", "bf16"])
@pytest.mark.parametrize("shape", UMMA_SK_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_tensor_core_split_tiles(mode, shape):
    m, n, k = shape
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert tgemm.tgemm_plan(mode, m, n, k, sm)["stream_k"]   # this device takes stream-K here
    parity.full_check(mode, inputs.random_case(9000 + m + n + k, m, n, k, kind="int"), f"{mode} int {shape}")
    case = inputs.random_case(9500 + m + n + k, m, n, k, kind="uniform")
    parity.full_check(mode, case, f"{mode} uniform {shape}")
    A, B = parity.inputs_for(mode, case)
    A, B = parity.to_device(A), parity.to_device(B)
    assert torch.equal(parity.ENTRY[mode](A, B), parity.ENTRY[mode](A, B))


# Extremes of k: 4096 k-phases on 4 tiles (the fp32 path splits them 8 ways,
# 512 phases per piece; integer sums reach 2^20, still exact in fp32), and a
# single k-phase over a large ragged output.
EXTREME_K_SHAPES = [(256, 256, 65536), (4100, 8200, 16)]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("shape", EXTREME_K_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_extreme_k(mode, shape):
    m, n, k = shape
    parity.full_check(mode, inputs.random_case(9900 + m + n + k, m, n, k, kind="int"), f"{mode} int {shape}")


@pytest.mark.parametrize("mode", MODES)
def test_leading_dimensions_and_untouched_padding(mode):
    m, n, k = 200, 150, 90
    case = inputs.random_case(4242, m, n, k, kind="int")
    A_np, B_np = parity.inputs_for(mode, case)
    dtype = torch.bfloat16 if mode == "bf16" else torch.float32
    A_big = torch.zeros((m, k + 13), dtype=dtype, device="cuda")
    B_big = torch.zeros((k, n + 6), dtype=dtype, device="cuda")
    A_big[:, 5:5 + k] = parity.to_device(A_np)
    B_big[:, :n] = parity.to_device(B_np)
    C_big = torch.full((m, n + 10), float("nan"), device="cuda")
    A, B, C = A_big[:, 5:5 + k], B_big[:, :n], C_big[:, 3:3 + n]
    parity.ENTRY[mode](A, B, C)
    torch.cuda.synchronize()
    P, D = oracle.gemm(A_np, B_np)
    parity.check(mode, C.cpu().numpy(), P, D, True, f"{mode} strided")
    host = C_big.cpu().numpy()
    assert np.all(np.isnan(host[:, :3])) and np.all(np.isnan(host[:, 3 + n:])), "wrote outside C"


@pytest.mark.parametrize("mode", MODES)
def test_k_zero_gives_zeros(mode):
    dtype = torch.bfloat16 if mode == "bf16" else torch.float32
    A = torch.empty((7, 0), dtype=dtype, device="cuda")
    B = torch.empty((0, 5), dtype=dtype, device="cuda")
    C = torch.full((7, 5), 3.0, device="cuda")
    parity.ENTRY[mode](A, B, C)
    torch.cuda.synchronize()
    assert torch.all(C == 0)


@pytest.mark.parametrize("mode", MODES)
def test_repeat_runs_are_bit_identical(mode):
    case = inputs.random_case(555, 1000, 700, 900, kind="normal")
    A_np, B_np = parity.inputs_for(mode, case)
    A, B = parity.to_device(A_np), parity.to_device(B_np)
    c1 = parity.ENTRY[mode](A, B)
    c2 = parity.ENTRY[mode](A, B)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)


def test_tf32_input_conversion(capsys):
    """How the tensor core reduces fp32 operands to TF32 (the pages are silent):
    the product agrees with the oracle on inputs reduced one way to within fp32
    accumulation error, and with the other only to TF32 precision."""
    m, n, k = 256, 256, 1024
    case = inputs.random_case(4343, m, n, k, kind="uniform")
    C = parity.run("tf32", case.A, case.B).cpu().numpy().astype(np.float64)
    errs = {}
    for conv in ("trunc", "rne"):
        P, D = oracle.gemm(inputs.to_tf32(case.A, conv), inputs.to_tf32(case.B, conv))
        errs[conv] = float(np.max(np.abs(C - P) / D))
    best = min(errs, key=errs.get)
    other = "rne" if best == "trunc" else "trunc"
    with capsys.disabled():
        print(f"\nTF32 operand conversion: {best} (max error {errs[best]:.2e}; {other}: {errs[other]:.2e})")
    assert errs[best] <= 1e-5, errs
    assert errs[other] > 10 * errs[best], errs
    # Measured on GB300: truncation (5.8e-7 against the truncated-input oracle, 1.35e-4 against RNE).
    assert best == "trunc", errs


def _boundary_shapes(count, seed, budget=1.2e9):
    """Seeded shapes that sit near the dispatch boundaries: m around 64 (the
    skinny bf16 kernel), sizes around multiples of 64/128/224/256 (tile edges),
    k around 1024, 2048 and 3072 (the tensor-core tiles are 256 rows high from
    k = 3072, and from k = 1024 where those rounds fill as well) and
    tile counts around multiples of 152 (a partly empty last wave: split
    pieces, 224-wide tiles, stream-K)."""
    rng = np.random.default_rng(seed)
    near = lambda base: int(max(1, base + rng.integers(-3, 4)))
    out = []
    while len(out) < count:
        m = near(int(rng.choice([1, 16, 32, 48, 64, 65, 128, 256, 1024, 1536, 2048, 2432, 3072])))
        n = near(int(rng.choice([8, 64, 128, 224, 256, 448, 896, 1536, 2048, 2432, 3072])))
        k = near(int(rng.choice([1, 16, 64, 129, 1024, 2048, 2049, 3072, 3100])))
        if m * n * k <= budget:
            out.append((m, n, k))
    return out


@pytest.mark.parametrize("shape", _boundary_shapes(36, 2024), ids=lambda s: "x".join(map(str, s)))
def test_boundary_shapes_exact(shape):
    m, n, k = shape
    case = inputs.random_case(31 * m + 7 * n + k, m, n, k, kind="int")
    for mode in MODES:
        parity.full_check(mode, case, f"{mode} int {shape}")


def _sampled_check(mode, case, n_rows, n_entries, seed):
    A_np, B_np = parity.inputs_for(mode, case)
    C = parity.run(mode, A_np, B_np)
    m, n = C.shape
    rng = np.random.default_rng(seed)
    rows = sorted(set([0, 1, 127, 128, 129, m // 2, m - 1] + rng.integers(0, m, n_rows).tolist()))
    Csub = C[torch.tensor(rows, device=C.device)].cpu().numpy()
    P, D = oracle.gemm(A_np[rows], B_np)
    err_rows = parity.check(mode, Csub, P, D, case.exact, f"{mode} {case} rows")
    ri = rng.integers(0, m, n_entries)
    ci = rng.integers(0, n, n_entries)
    Pe, De = oracle.gemm_entries(A_np, B_np, ri, ci)
    got = C[torch.from_numpy(ri).to(C.device), torch.from_numpy(ci).to(C.device)].cpu().numpy()
    err_ent = parity.check(mode, got.reshape(-1, 1), Pe.reshape(-1, 1), De.reshape(-1, 1), case.exact,
                           f"{mode} {case} entries")
    return max(err_rows, err_ent)


@pytest.fixture(scope="module")
def case_n4096():
    return inputs.make("n4096")


@pytest.mark.parametrize("mode", ["f32", "tf32"])
def test_full_size_4096_fp32(mode, case_n4096):
    _sampled_check(mode, case_n4096, 24, 2000, 11)


def test_full_size_8192_bf16():
    _sampled_check("bf16", inputs.make("bf16_8192"), 8, 1000, 12)


def test_skinny_16x8192x8192_bf16():
    parity.full_check("bf16", inputs.make("skinny"))


# bf16 with m <= 64 takes the transposed cluster kernel: 16-, 32- and 64-row
# forms (m <= 16, <= 32, <= 64), k split over 1..8 CTAs of a cluster, ragged
# column tiles and k tails, and a k-slice count that does not divide k.
SKINNY_SHAPES = [(16, 128, 64), (17, 300, 200), (24, 1000, 4100), (32, 1000, 8192), (33, 129, 70),
                 (48, 2000, 1000), (63, 8200, 130), (64, 4096, 8192), (3, 20000, 4160)]


@pytest.mark.parametrize("shape", SKINNY_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_skinny_bf16_row_forms(shape):
    m, n, k = shape
    parity.full_check("bf16", inputs.random_case(5000 + m + 7 * n + 13 * k, m, n, k, kind="int"),
                      f"bf16 skinny int {shape}")
    parity.full_check("bf16", inputs.random_case(6000 + m + 7 * n + 13 * k, m, n, k, kind="normal"),
                      f"bf16 skinny normal {shape}")


# One very large extent at a time (the other two small): grid and tile
# indices far beyond the other tests, TMA coordinates into the millions, and
# the skinny kernel with 65536 column tiles.  Checked element by element.
LARGE_EXTENT_SHAPES = [(1, 8388608, 16), (1048576, 8, 32), (3000, 3, 20000), (64, 2097152, 16)]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("shape", LARGE_EXTENT_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_large_single_extent(mode, shape):
    m, n, k = shape
    parity.full_check(mode, inputs.random_case(7000 + m % 997 + 7 * (n % 991) + 13 * k, m, n, k, kind="int"),
                      f"{mode} int {shape}")


def _strided_cases(count, seed):
    """Seeded shapes, each operand a view into a larger buffer: a random row
    padding (leading dimension = extent + 0..9) and a random base offset of
    0..3 elements, so every combination of 16-byte-aligned and misaligned
    operands and C appears (re-pitch, vector and scalar epilogue stores)."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        m, n, k = (int(x) for x in rng.integers(1, 700, 3))
        pads = tuple(int(x) for x in rng.integers(0, 10, 3))
        offs = tuple(int(x) for x in rng.integers(0, 4, 3))
        out.append((m, n, k, pads, offs))
    return out


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("case_spec", _strided_cases(12, 4711), ids=lambda c: "x".join(map(str, c[:3])))
def test_random_views_exact_and_nothing_written_outside_c(mode, case_spec):
    m, n, k, (pa, pb, pc), (oa, ob, oc) = case_spec
    case = inputs.random_case(17 * m + 5 * n + k, m, n, k, kind="int")
    A_np, B_np = parity.inputs_for(mode, case)
    dtype = torch.bfloat16 if mode == "bf16" else torch.float32
    A_buf = torch.zeros(oa + m * (k + pa), dtype=dtype, device="cuda")
    B_buf = torch.zeros(ob + k * (n + pb), dtype=dtype, device="cuda")
    C_buf = torch.full((oc + m * (n + pc) + 8,), float("nan"), device="cuda")
    A = A_buf[oa:oa + m * (k + pa)].view(m, k + pa)[:, :k]
    B = B_buf[ob:ob + k * (n + pb)].view(k, n + pb)[:, :n]
    C = C_buf[oc:oc + m * (n + pc)].view(m, n + pc)[:, :n]
    A.copy_(parity.to_device(A_np))
    B.copy_(parity.to_device(B_np))
    parity.ENTRY[mode](A, B, C)
    torch.cuda.synchronize()
    P, D = oracle.gemm(A_np, B_np)
    parity.check(mode, C.cpu().numpy(), P, D, True, f"{mode} view {case_spec}")
    host = C_buf.cpu().numpy()
    inside = np.zeros(host.shape, dtype=bool)
    for i in range(m):
        inside[oc + i * (n + pc): oc + i * (n + pc) + n] = True
    assert np.all(np.isnan(host[~inside])), "wrote outside C"


# C with 16-byte aligned rows (the tensor-core paths store it with TMA) and a
# right edge in every position within a 16-byte granule: nothing may be
# written past column n - 1 (a TMA store clips rows at 16-byte granularity,
# so a ragged edge block must not take it).
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("n", [657, 658, 659, 660, 33, 250])
def test_ragged_right_edge_with_aligned_rows(mode, n):
    m, k = 300, 200
    case = inputs.random_case(4242 + n, m, n, k, kind="int")
    A_np, B_np = parity.inputs_for(mode, case)
    ldc = (n + 3) // 4 * 4 + 4                      # 16-byte pitch, at least 4 guard columns
    C_buf = torch.full(((m + 1) * ldc,), float("nan"), device="cuda")
    C = C_buf[: m * ldc].view(m, ldc)[:, :n]
    parity.ENTRY[mode](parity.to_device(A_np), parity.to_device(B_np), C)
    torch.cuda.synchronize()
    P, D = oracle.gemm(A_np, B_np)
    parity.check(mode, C.cpu().numpy(), P, D, True, f"{mode} ragged edge n={n}")
    host = C_buf.view(m + 1, ldc).cpu().numpy()
    assert np.all(np.isnan(host[:m, n:])), f"{mode}: wrote past column {n - 1}"
    assert np.all(np.isnan(host[m:])), f"{mode}: wrote past row {m - 1}"


# bf16 128-row tiles as multicast CTA pairs (128-row tiles, no stream-K region,
# an even number of tile rows and at least two rounds of tiles on GB300): whole
# output against the oracle, exact sizes, ragged m / n / k (the last tile row
# partly empty) and short k.
PAIR_SHAPES = [(2048, 4864, 1000), (2000, 4800, 999), (4096, 2432, 200), (1536, 9728, 1024)]


def takes_pairs(m, n, k, sms=152):
    """The launcher's choice, restated (launch_rules.pairs) and checked against
    the library's own plan (tgemm_plan)."""
    want = launch_rules.pairs(m, n, k, sms)
    assert tgemm.tgemm_plan("bf16", m, n, k, sms)["pairs"] == want
    return want


def test_pair_rule_restatement():
    assert takes_pairs(2048, 4864, 1000) and takes_pairs(1536, 9728, 1024)
    assert not takes_pairs(8192, 8192, 2048)        # 256-row tiles fill its rounds as well
    assert not takes_pairs(4097, 3001, 1023)        # 33 tile rows
    assert not takes_pairs(2560, 4352, 1024)        # stream-K: 340 tiles fill 75 % of 3 rounds
    assert not takes_pairs(8192, 8192, 8192)        # 256-row tiles


@pytest.mark.parametrize("shape", PAIR_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_bf16_cta_pairs(shape):
    m, n, k = shape
    assert takes_pairs(m, n, k)
    parity.full_check("bf16", inputs.random_case(8100 + m + n + k, m, n, k, kind="int"), f"bf16 pairs int {shape}")
    parity.full_check("bf16", inputs.random_case(8200 + m + n + k, m, n, k, kind="normal"),
                      f"bf16 pairs normal {shape}")


def test_bf16_cta_pairs_with_unaligned_c():
    """Pairs with C that TMA cannot describe (row pitch n + 1): the pair kernel
    with eight epilogue warps on the read-back path; NaN guard columns must
    stay untouched."""
    m, n, k = 2048, 4864, 1000
    assert takes_pairs(m, n, k)
    case = inputs.random_case(8300, m, n, k, kind="int")
    A_np, B_np = parity.inputs_for("bf16", case)
    ldc = n + 1
    C_buf = torch.full((m * ldc + 8,), float("nan"), device="cuda")
    C = C_buf[: m * ldc].view(m, ldc)[:, :n]
    parity.ENTRY["bf16"](parity.to_device(A_np), parity.to_device(B_np), C)
    torch.cuda.synchronize()
    P, D = oracle.gemm(A_np, B_np)
    parity.check("bf16", C.cpu().numpy(), P, D, True, "bf16 pairs, unaligned C")
    host = C_buf[: m * ldc].view(m, ldc).cpu().numpy()
    assert np.all(np.isnan(host[:, n:])), "wrote past column n - 1"
    assert np.all(np.isnan(C_buf[m * ldc:].cpu().numpy()))


# Fewer tensor-core tiles than SMs with long k: each tile is cut along k into
# split-K pieces (one CTA each, partial sums in the workspace) that the reduce
# kernel adds in piece order.  256-row and 128-row tiles, ragged edges, m just
# above the skinny kernel's 64 rows.  Whole output against the oracle, and
# repeated runs bit-identical.
PIECE_SHAPES = [(1024, 1024, 8192), (65, 4096, 4096), (1000, 1001, 2000), (129, 1000, 3072)]


@pytest.mark.parametrize("mode", ["tf32", "bf16"])
@pytest.mark.parametrize("shape", PIECE_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_split_k_pieces(mode, shape):
    m, n, k = shape
    assert launch_rules.pieces(m, n, k, mode) >= 2
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert tgemm.tgemm_plan(mode, m, n, k, sm)["pieces"] >= 2
    parity.full_check(mode, inputs.random_case(8400 + m + n + k, m, n, k, kind="int"), f"{mode} pieces int {shape}")
    case = inputs.random_case(8500 + m + n + k, m, n, k, kind="uniform")
    parity.full_check(mode, case, f"{mode} pieces uniform {shape}")
    A, B = parity.inputs_for(mode, case)
    A, B = parity.to_device(A), parity.to_device(B)
    assert torch.equal(parity.ENTRY[mode](A, B), parity.ENTRY[mode](A, B))


@pytest.mark.parametrize("mode", ["tf32", "bf16"])
def test_split_k_pieces_with_unaligned_c(mode):
    """Pieces with C rows that are not 16-byte aligned (row pitch n + 1): the
    reduce kernel's scalar stores; NaN guard columns must stay untouched."""
    m, n, k = 1000, 1001, 2000
    assert launch_rules.pieces(m, n, k, mode) >= 2
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert tgemm.tgemm_plan(mode, m, n, k, sm)["pieces"] >= 2
    case = inputs.random_case(8600, m, n, k, kind="int")
    A_np, B_np = parity.inputs_for(mode, case)
    ldc = n + 1
    C_buf = torch.full((m * ldc + 8,), float("nan"), device="cuda")
    C = C_buf[: m * ldc].view(m, ldc)[:, :n]
    parity.ENTRY[mode](parity.to_device(A_np), parity.to_device(B_np), C)
    torch.cuda.synchronize()
    P, D = oracle.gemm(A_np, B_np)
    parity.check(mode, C.cpu().numpy(), P, D, True, f"{mode} pieces, unaligned C")
    host = C_buf[: m * ldc].view(m, ldc).cpu().numpy()
    assert np.all(np.isnan(host[:, n:])), "wrote past column n - 1"
    assert np.all(np.isnan(C_buf[m * ldc:].cpu().numpy()))
