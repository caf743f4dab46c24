"""Seeded synthetic inputs for the tiled matrix multiply.

This module only draws numbers: it holds none of the product's arithmetic and
imports neither the CUDA path nor the oracle, so both may consume what it
makes.  Every matrix is a pure function of ``(seed, stream, shape)``.

Generator
    SplitMix64 used in counter mode: draw ``i`` of stream ``s`` under seed
    ``seed`` is ``mix64(key + (i + 1) * GAMMA)`` with
    ``key = mix64(seed * GAMMA + s)``, ``GAMMA = 0x9E3779B97F4A7C15`` and
    ``mix64`` the SplitMix64 finaliser (Steele, Lea and Flood, "Fast
    splittable pseudorandom number generators", OOPSLA 2014), all modulo 2^64.

Distributions (each element consumes one 64-bit draw, Box-Muller two)
    uniform [-1, 1]  : top 24 bits r, value (2r + 1 - 2^24) / 2^24 (exact in fp32)
    integers lo..hi  : top 32 bits r, value lo + floor(r * (hi - lo + 1) / 2^32)
    normal N(0, 1)   : Box-Muller in double from two draws, times a scale,
                       rounded to fp32
    bf16             : fp32 values rounded to nearest-even bf16 bit patterns

Workloads (seed 1000 + c for workload c; M is stream 0, N is stream 1)
    worked_4x4  : M(i,k) = 4i + k + 1, N(k,j) = 16 - (4k + j)  (4x4, tile 2)
    int64       : 64^3, integers in [-3, 3]
    u128        : 128^3, uniform [-1, 1]
    int1024     : 1024^3, integers in [-4, 4]
    n4096       : 4096^3, N(0, 1)
    bf16_8192   : 8192^3 bf16, N(0, 1) / sqrt(8192)
    irregular   : 4097 x 3001 x 1023, uniform [-1, 1], lda = 1023, ldb = 3001
    skinny      : 16 x 8192 x 8192 bf16, uniform [-1, 1]
    long_k      : 1024 x 1024 x 8192, uniform [-1, 1] (fewer output tiles than SMs)
"""
from __future__ import annotations

import math

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_MASK64 = (1 << 64) - 1
_CHUNK = 1 << 22


def _mix64_int(z: int) -> int:
    z &= _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * np.uint64(0xBF58476D1CE4E5B9)
    z = z ^ (z >> np.uint64(27))
    z = z * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, stream: int) -> int:
    return _mix64_int((seed * 0x9E3779B97F4A7C15 + stream) & _MASK64)


def draws(seed: int, stream: int, count: int, offset: int = 0) -> np.ndarray:
    """``count`` raw 64-bit draws of ``(seed, stream)`` starting at draw ``offset``."""
    return draws_from_key(stream_key(seed, stream), count, offset)


def draws_from_key(key: int, count: int, offset: int = 0) -> np.ndarray:
    """SplitMix64 outputs ``offset .. offset+count-1`` of a generator whose state starts at ``key``."""
    key = np.uint64(key & _MASK64)
    out = np.empty(count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        for lo in range(0, count, _CHUNK):
            hi = min(count, lo + _CHUNK)
            idx = np.arange(offset + lo + 1, offset + hi + 1, dtype=np.uint64)
            out[lo:hi] = _mix64(key + idx * GAMMA)
    return out


def uniform_pm1(seed: int, stream: int, shape) -> np.ndarray:
    """Uniform values in (-1, 1), each an exact fp32 (odd multiple of 2^-24)."""
    count = int(np.prod(shape))
    out = np.empty(count, dtype=np.float32)
    for lo in range(0, count, _CHUNK):
        hi = min(count, lo + _CHUNK)
        r = (draws(seed, stream, hi - lo, lo) >> np.uint64(40)).astype(np.int64)
        out[lo:hi] = ((2 * r + 1 - (1 << 24)).astype(np.float64) * 2.0 ** -24).astype(np.float32)
    return out.reshape(shape)


def integers(seed: int, stream: int, shape, lo: int, hi: int) -> np.ndarray:
    """Integers uniform in ``lo..hi`` (inclusive), stored as fp32."""
    count = int(np.prod(shape))
    span = np.uint64(hi - lo + 1)
    out = np.empty(count, dtype=np.float32)
    with np.errstate(over="ignore"):
        for a in range(0, count, _CHUNK):
            b = min(count, a + _CHUNK)
            r = draws(seed, stream, b - a, a) >> np.uint64(32)
            out[a:b] = ((r * span) >> np.uint64(32)).astype(np.int64) + lo
    return out.reshape(shape)


def normal(seed: int, stream: int, shape, scale: float = 1.0) -> np.ndarray:
    """Normal values with standard deviation ``scale``, rounded to fp32.

    Element ``e`` uses draws ``2e`` and ``2e+1``: ``u1 = (d >> 11 + 1) / 2^53`` in
    (0, 1], ``u2 = (d >> 11) / 2^53``, value ``sqrt(-2 ln u1) cos(2 pi u2) * scale``.
    """
    count = int(np.prod(shape))
    out = np.empty(count, dtype=np.float32)
    for a in range(0, count, _CHUNK):
        b = min(count, a + _CHUNK)
        d = draws(seed, stream, 2 * (b - a), 2 * a).reshape(-1, 2) >> np.uint64(11)
        u1 = (d[:, 0].astype(np.float64) + 1.0) * 2.0 ** -53
        u2 = d[:, 1].astype(np.float64) * 2.0 ** -53
        out[a:b] = (np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2) * scale).astype(np.float32)
    return out.reshape(shape)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest bf16 (ties to even); returns uint16 bit patterns."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (bits + np.uint64(0x7FFF) + ((bits >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return rounded.astype(np.uint16)


def to_tf32(x: np.ndarray, mode: str = "rne") -> np.ndarray:
    """fp32 values reduced to TF32 precision (10 stored mantissa bits), still as
    float32: the low 13 mantissa bits cleared ("trunc") or rounded to nearest,
    ties to even ("rne").  Finite inputs only."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    if mode == "rne":
        bits = bits + np.uint64(0xFFF) + ((bits >> np.uint64(13)) & np.uint64(1))
    elif mode != "trunc":
        raise ValueError(mode)
    bits = bits & np.uint64(0xFFFFE000)
    return bits.astype(np.uint32).view(np.float32)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact fp32 values of bf16 bit patterns."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


class Case:
    """One synthetic problem: ``A`` is m x k, ``B`` is k x n, both row-major.

    ``dtype`` is ``"f32"`` (fp32 arrays) or ``"bf16"`` (uint16 bit patterns).
    ``lda``/``ldb``/``ldc`` are the leading dimensions the problem is quoted with.
    """

    def __init__(self, name, A, B, dtype, lda=None, ldb=None, ldc=None, exact=False):
        self.name = name
        self.A = A
        self.B = B
        self.dtype = dtype
        self.m, self.k = A.shape
        self.n = B.shape[1]
        self.lda = lda if lda is not None else max(self.k, 1)
        self.ldb = ldb if ldb is not None else max(self.n, 1)
        self.ldc = ldc if ldc is not None else max(self.n, 1)
        self.exact = exact

    @property
    def flops(self) -> int:
        return 2 * self.m * self.n * self.k

    def __repr__(self):
        return f"Case({self.name}: {self.m}x{self.n}x{self.k} {self.dtype})"


def worked_4x4() -> Case:
    i = np.arange(4).reshape(4, 1)
    k = np.arange(4).reshape(1, 4)
    M = (4 * i + k + 1).astype(np.float32)
    N = (16 - (4 * np.arange(4).reshape(4, 1) + np.arange(4).reshape(1, 4))).astype(np.float32)
    return Case("worked_4x4", M, N, "f32", exact=True)


def make(name: str, dtype: str | None = None) -> Case:
    """Build a named workload (see the module docstring)."""
    if name == "worked_4x4":
        c = worked_4x4()
    elif name == "int64":
        c = Case(name, integers(1000, 0, (64, 64), -3, 3), integers(1000, 1, (64, 64), -3, 3),
                 "f32", exact=True)
    elif name == "u128":
        c = Case(name, uniform_pm1(1000, 0, (128, 128)), uniform_pm1(1000, 1, (128, 128)), "f32")
    elif name == "int1024":
        c = Case(name, integers(1001, 0, (1024, 1024), -4, 4), integers(1001, 1, (1024, 1024), -4, 4),
                 "f32", exact=True)
    elif name == "n4096":
        c = Case(name, normal(1002, 0, (4096, 4096)), normal(1002, 1, (4096, 4096)), "f32")
    elif name == "bf16_8192":
        s = 1.0 / math.sqrt(8192)
        c = Case(name, to_bf16_bits(normal(1003, 0, (8192, 8192), s)),
                 to_bf16_bits(normal(1003, 1, (8192, 8192), s)), "bf16")
    elif name == "irregular":
        c = Case(name, uniform_pm1(1004, 0, (4097, 1023)), uniform_pm1(1004, 1, (1023, 3001)), "f32")
    elif name == "skinny":
        c = Case(name, to_bf16_bits(uniform_pm1(1004, 2, (16, 8192))),
                 to_bf16_bits(uniform_pm1(1004, 3, (8192, 8192))), "bf16")
    elif name == "long_k":
        c = Case(name, uniform_pm1(1005, 0, (1024, 8192)), uniform_pm1(1005, 1, (8192, 1024)), "f32")
    else:
        raise KeyError(f"unknown workload {name!r}")
    if dtype is not None and dtype != c.dtype:
        c = convert(c, dtype)
    return c


def convert(c: Case, dtype: str) -> Case:
    """The same values in another storage type (fp32 -> bf16 rounds to nearest even)."""
    if dtype == c.dtype:
        return c
    if dtype == "bf16":
        return Case(c.name, to_bf16_bits(c.A), to_bf16_bits(c.B), "bf16", c.lda, c.ldb, c.ldc,
                    exact=c.exact)
    if dtype == "f32":
        return Case(c.name, bf16_bits_to_f32(c.A), bf16_bits_to_f32(c.B), "f32", c.lda, c.ldb, c.ldc,
                    exact=c.exact)
    raise ValueError(dtype)


def random_case(seed: int, m: int, n: int, k: int, dtype: str = "f32", kind: str = "uniform") -> Case:
    """Ad-hoc problem of any shape (edge-tile sweeps)."""
    if kind == "uniform":
        A, B = uniform_pm1(seed, 0, (m, k)), uniform_pm1(seed, 1, (k, n))
    elif kind == "int":
        A, B = integers(seed, 0, (m, k), -4, 4), integers(seed, 1, (k, n), -4, 4)
    elif kind == "normal":
        A, B = normal(seed, 0, (m, k)), normal(seed, 1, (k, n))
    else:
        raise ValueError(kind)
    c = Case(f"rand{seed}_{m}x{n}x{k}", A, B, "f32", exact=(kind == "int"))
    return convert(c, dtype)
