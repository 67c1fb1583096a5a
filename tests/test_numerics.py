"""CPU checks of the numerical building blocks the kernels use.

The tensor-core kernels split an fp32 value x into hi = tf32(x) and
lo = tf32(x - hi), with tf32() = round to 10 explicit mantissa bits, to
nearest, ties away from zero, computed on the bit pattern as
(bits + 0x1000) & 0xFFFFE000. These tests pin that formula to an independent
definition (exact rational arithmetic) and check the error of the split that
the FP32-class bound relies on.
"""

from fractions import Fraction

import numpy as np

import synth


def tf32_bits_formula(x: np.ndarray) -> np.ndarray:
    u = x.astype(np.float32).view(np.uint32)
    return ((u.astype(np.uint64) + 0x1000) & 0xFFFFE000).astype(np.uint32).view(np.float32)


def tf32_exact(v: float) -> float:
    """Round v (finite, normal) to 11 significant bits, ties away from zero."""
    if v == 0:
        return 0.0
    f = Fraction(v)
    mag = abs(f)
    e = 0
    while mag >= 2:
        mag /= 2
        e += 1
    while mag < 1:
        mag *= 2
        e -= 1
    scaled = mag * 1024  # 11 significant bits: 1.xxxxxxxxxx
    q, r = divmod(scaled.numerator, scaled.denominator)
    if 2 * r >= scaled.denominator:  # ties away from zero
        q += 1
    out = Fraction(q, 1024) * Fraction(2) ** e
    return float(out if f > 0 else -out)


def test_rounding_formula_matches_exact_rounding():
    vals = np.concatenate([
        synth.normal((3000,), 5),
        synth.uniform_pm1((3000,), 6) * 1e-3,
        synth.uniform_pm1((1000,), 7) * 3e4,
        # exact ties: 11 significant bits plus a trailing half unit
        np.array([1 + 2.0 ** -11, -(1 + 2.0 ** -11), 1.5 + 2.0 ** -11, 1 + 3 * 2.0 ** -11,
                  2 - 2.0 ** -12, -(2 - 2.0 ** -12), 1 + 2.0 ** -11 - 2.0 ** -23], dtype=np.float32),
    ]).astype(np.float32)
    got = tf32_bits_formula(vals)
    for v, gv in zip(vals.tolist(), got.tolist()):
        assert gv == tf32_exact(v), (v, gv, tf32_exact(v))
        assert np.float32(gv).view(np.uint32) & 0x1FFF == 0


def test_split_error():
    # hi + lo reproduces x to within 2^-22 |x| (lo itself rounded to TF32),
    # and each part is a TF32 value
    x = np.concatenate([synth.normal((20000,), 9), synth.uniform_pm1((20000,), 10)]).astype(np.float32)
    hi = tf32_bits_formula(x)
    lo = tf32_bits_formula((x - hi).astype(np.float32))
    assert np.all(hi.view(np.uint32) & 0x1FFF == 0) and np.all(lo.view(np.uint32) & 0x1FFF == 0)
    # x - hi is exact in fp32
    assert np.all((x.astype(np.float64) - hi.astype(np.float64)) == (x - hi).astype(np.float64))
    err = np.abs(x.astype(np.float64) - hi.astype(np.float64) - lo.astype(np.float64))
    assert np.all(err <= 2.0 ** -22 * np.abs(x.astype(np.float64)))
