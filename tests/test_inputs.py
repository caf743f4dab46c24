"""The seeded input generators shared by the oracle side and the CUDA side."""
import numpy as np
import pytest
import torch

from dense_tiled_matrix_gb300 import inputs as I


def test_splitmix64_published_vector():
    # SplitMix64 started at state 1234567: the first outputs of the reference
    # generator (Steele, Lea, Flood 2014; Vigna's splitmix64.c).
    got = I.draws_from_key(1234567, 3)
    assert got.tolist() == [6457827717110365317, 3203168211198807973, 9817491932198370423]


def test_counter_mode_offsets_and_chunks(monkeypatch):
    full = I.draws(7, 3, 100)
    assert np.array_equal(full[37:], I.draws(7, 3, 63, offset=37))
    monkeypatch.setattr(I, "_CHUNK", 16)
    assert np.array_equal(full, I.draws(7, 3, 100))
    u = I.uniform_pm1(7, 3, (10, 10))
    monkeypatch.setattr(I, "_CHUNK", 1 << 22)
    assert np.array_equal(u, I.uniform_pm1(7, 3, (10, 10)))


def test_streams_and_seeds_differ():
    a = I.draws(1000, 0, 8)
    assert not np.array_equal(a, I.draws(1000, 1, 8))
    assert not np.array_equal(a, I.draws(1001, 0, 8))


def test_uniform_is_exact_and_in_range():
    u = I.uniform_pm1(11, 0, (256, 256))
    assert u.dtype == np.float32
    assert np.all(np.abs(u) < 1.0)
    scaled = u.astype(np.float64) * 2.0 ** 24
    assert np.all(scaled == np.round(scaled)) and np.all(np.mod(scaled, 2) == 1)
    assert abs(float(u.mean())) < 0.01


def test_integers_cover_range():
    v = I.integers(12, 0, (100, 100), -4, 4)
    assert set(np.unique(v).tolist()) == set(range(-4, 5))
    counts = np.unique(v, return_counts=True)[1]
    assert counts.min() > 0.8 * counts.mean()


def test_normal_moments():
    x = I.normal(13, 0, (512, 512))
    assert abs(float(x.mean())) < 0.01 and abs(float(x.std()) - 1.0) < 0.01
    y = I.normal(13, 0, (512, 512), scale=0.5)
    assert np.allclose(y, (x.astype(np.float64) * 0.5).astype(np.float32), rtol=1e-6, atol=0)


def test_bf16_rounding_matches_torch():
    vals = np.concatenate([
        I.normal(14, 0, (4096,)),
        np.array([1.0, 1.00390625, 1.01171875, -1.00390625, 0.0, -0.0, 3.0e38, 1e-40],
                 dtype=np.float32)])
    bits = I.to_bf16_bits(vals)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bits, ref)
    back = I.bf16_bits_to_f32(bits)
    assert np.array_equal(back, torch.from_numpy(vals).to(torch.bfloat16).float().numpy())


def test_named_workloads_small():
    c = I.make("worked_4x4")
    assert c.A[0].tolist() == [1, 2, 3, 4] and c.B[:, 0].tolist() == [16, 12, 8, 4]
    for name, shape in [("int64", (64, 64, 64)), ("u128", (128, 128, 128))]:
        c = I.make(name)
        assert (c.m, c.n, c.k) == shape
        assert np.array_equal(c.A, I.make(name).A)
    assert set(np.unique(I.make("int64").A).tolist()) <= set(range(-3, 4))
    cb = I.make("u128", "bf16")
    assert cb.A.dtype == np.uint16 and cb.dtype == "bf16"


def test_tf32_reduction():
    one = 1.0
    ulp = 2.0 ** -10                      # TF32 spacing at 1
    vals = np.array([one + ulp / 2,       # exact tie: even neighbour is 1
                     one + ulp + ulp / 2, # tie: rounds up to 1 + 2 ulp (even)
                     one + ulp / 2 + 2.0 ** -20,   # above the tie
                     -(one + 3 * ulp / 4),
                     3.0, 2.0 ** -100], dtype=np.float32)
    rne = I.to_tf32(vals, "rne")
    trunc = I.to_tf32(vals, "trunc")
    assert rne.tolist() == [1.0, one + 2 * ulp, one + ulp, -(one + ulp), 3.0, 2.0 ** -100]
    assert trunc.tolist() == [1.0, one + ulp, 1.0, -1.0, 3.0, 2.0 ** -100]
    # 10 stored mantissa bits: the low 13 bits of every result are zero
    r = I.to_tf32(I.uniform_pm1(5, 0, (1000,)), "rne")
    assert not (r.view(np.uint32) & 0x1FFF).any()
