"""Seeded synthetic inputs for the fp32 GEMM C = A x B.

This module only draws numbers. It holds none of the product's arithmetic, so
both the fp64 oracle (``oracle/``) and the CUDA library's tests and benchmark
take their operands from here and from nowhere else.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014; the finaliser constants are the ones Vigna
published for ``splitmix64.c``), used as a counter-based generator: the value
for linear index ``i`` under ``seed`` is the SplitMix64 output for the state
``seed + (i + 1) * 0x9E3779B97F4A7C15 (mod 2**64)``.  Every element is
therefore a pure function of (seed, index): identical on every machine and
independent of how a matrix is later tiled or sharded.

Distributions (the pages ask for random inputs but fix none; the workloads
below use the shapes and distributions of the benchmark configurations):

* ``uniform_pm1``: ``u = (r >> 40) * 2**-24`` and ``x = 2u - 1``.  Every value
  is a multiple of 2**-23 in [-1, 1), hence exact in fp32.
* ``normal``: Box-Muller in fp64 on pairs of draws, rounded once to fp32.
* ``small_integers``: integer values in [lo, hi]; products and sums of such
  values stay exact in fp32 and TF32 as long as partial sums stay below 2**24.
"""

from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Workload table: the five benchmark configurations (the fifth has two
# shapes). Row-major, dense leading dimensions, C overwritten.
CONFIGS = {
    "c1": dict(M=512, N=512, K=512, dist="uniform", seed_a=1002, seed_b=1003),
    "c2": dict(M=1024, N=1024, K=1024, dist="uniform", seed_a=1004, seed_b=1005),
    "c3": dict(M=2048, N=2048, K=2048, dist="uniform", seed_a=1006, seed_b=1007),
    "c4": dict(M=4096, N=4096, K=4096, dist="uniform", seed_a=1008, seed_b=1009),
    "c5a": dict(M=1000, N=1531, K=777, dist="normal", seed_a=1010, seed_b=1011),
    "c5b": dict(M=8192, N=11008, K=4096, dist="normal", seed_a=1010, seed_b=1011),
}


def splitmix64(seed: int, index: np.ndarray) -> np.ndarray:
    """SplitMix64 output for each counter in ``index`` (uint64 array)."""
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + (index.astype(np.uint64) + np.uint64(1)) * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def _count(shape) -> int:
    n = 1
    for s in shape:
        n *= int(s)
    return n


def uniform_pm1(shape, seed: int) -> np.ndarray:
    """fp32 array of ``shape`` with i.i.d. values on the grid 2**-23 * Z in [-1, 1)."""
    n = _count(shape)
    r = splitmix64(seed, np.arange(n, dtype=np.uint64))
    k = (r >> np.uint64(40)).astype(np.int64)           # 24 random bits
    x = (k - (1 << 23)).astype(np.float64) * 2.0 ** -23  # = 2u - 1, exact
    return x.astype(np.float32).reshape(shape)


def normal(shape, seed: int) -> np.ndarray:
    """fp32 array of ``shape`` with i.i.d. N(0, 1) values (Box-Muller on pairs)."""
    n = _count(shape)
    npair = (n + 1) // 2
    p = np.arange(npair, dtype=np.uint64)
    r1 = splitmix64(seed, np.uint64(2) * p)
    r2 = splitmix64(seed, np.uint64(2) * p + np.uint64(1))
    u1 = ((r1 >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53  # (0, 1]
    u2 = (r2 >> np.uint64(11)).astype(np.float64) * 2.0 ** -53          # [0, 1)
    rad = np.sqrt(-2.0 * np.log(u1))
    theta = 2.0 * np.pi * u2
    out = np.empty(2 * npair, dtype=np.float64)
    out[0::2] = rad * np.cos(theta)
    out[1::2] = rad * np.sin(theta)
    return out[:n].astype(np.float32).reshape(shape)


def small_integers(shape, seed: int, lo: int = -8, hi: int = 8) -> np.ndarray:
    """fp32 array of integer values drawn uniformly from [lo, hi]."""
    n = _count(shape)
    r = splitmix64(seed, np.arange(n, dtype=np.uint64))
    span = np.uint64(hi - lo + 1)
    v = (r % span).astype(np.int64) + lo
    return v.astype(np.float32).reshape(shape)


def draw(dist: str, shape, seed: int) -> np.ndarray:
    if dist == "uniform":
        return uniform_pm1(shape, seed)
    if dist == "normal":
        return normal(shape, seed)
    if dist == "int":
        return small_integers(shape, seed)
    raise ValueError(f"unknown distribution {dist!r}")


def config_operands(name: str):
    """(A, B, cfg) for a named workload; A is M x K and B is K x N, row-major fp32."""
    cfg = CONFIGS[name]
    a = draw(cfg["dist"], (cfg["M"], cfg["K"]), cfg["seed_a"])
    b = draw(cfg["dist"], (cfg["K"], cfg["N"]), cfg["seed_b"])
    return a, b, cfg


def embed_strided(x: np.ndarray, ld: int, fill: float = np.nan) -> np.ndarray:
    """Copy a rows x cols matrix into a buffer with leading dimension ``ld``.

    Returns the full padded 2-D buffer (rows x ld); the padding holds ``fill``
    so that a reader that strays into it produces NaN.
    """
    rows, cols = x.shape
    assert ld >= cols
    buf = np.full((rows, ld), fill, dtype=np.float32)
    buf[:, :cols] = x
    return buf
