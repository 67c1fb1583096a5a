"""Pins of the fp64 vector-sum oracle (oracle.vector_sum) to facts fixed
outside it: closed forms, exact integer arithmetic, brute force over Python
integers and fractions, and the integer self-test of "GPU compute shaders"
(section "Code": values (37 i mod 101) - 50 for i < 10000). A planted mistake
in a copy of the definition (a dropped element, a sign error, an absolute
value lost) must fail them."""

from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth


def pin_pages_integer_pattern(vsum):
    # the page's own check: integer values keep every f32 partial sum exact,
    # so the sum equals the exact integer sum
    n = 10_000
    v = np.array([(i * 37 % 101) - 50 for i in range(n)], dtype=np.float32)
    exact = sum((i * 37 % 101) - 50 for i in range(n))
    s, scale = vsum(v)
    assert s == exact
    assert scale == sum(abs((i * 37 % 101) - 50) for i in range(n))


def pin_closed_forms(vsum):
    for n in (0, 1, 7, 1000, 1 << 16):
        assert vsum(np.ones(n, np.float32)) == (n, n)
        r = np.arange(n, dtype=np.float32)
        assert vsum(r)[0] == n * (n - 1) // 2
        alt = np.where(np.arange(n) % 2 == 0, 1.0, -1.0).astype(np.float32)
        assert vsum(alt) == (n % 2, n)


def pin_brute_force(vsum):
    # exact rational sum of random fp32 values (every fp32 is a dyadic rational)
    for seed, n in ((1, 1), (2, 5), (3, 333), (4, 4099)):
        x = synth.normal((n,), 700 + seed).reshape(-1)
        exact = sum(Fraction(float(v)) for v in x)
        s, scale = vsum(x)
        assert abs(Fraction(s) - exact) <= Fraction(n) * Fraction(2) ** -52 * Fraction(scale)
        assert scale == pytest.approx(float(sum(abs(Fraction(float(v))) for v in x)), rel=1e-15)


PINS = [pin_pages_integer_pattern, pin_closed_forms, pin_brute_force]


@pytest.mark.parametrize("pin", PINS)
def test_oracle_sum_pins(pin):
    pin(oracle.vector_sum)


def _definition(x, drop=None, flip=None, lose_abs=False):
    s, scale = 0.0, 0.0
    for i, v in enumerate(x.astype(np.float64)):
        if i == drop:
            continue
        s += -v if i == flip else v
        scale += v if lose_abs else abs(v)
    return s, scale


@pytest.mark.parametrize("mutant", [dict(drop=0), dict(flip=3), dict(lose_abs=True)])
def test_planted_mistakes_fail_the_pins(mutant):
    def vsum(x):
        return _definition(np.asarray(x), **mutant)

    failed = 0
    for pin in PINS:
        try:
            pin(vsum)
        except AssertionError:
            failed += 1
    assert failed >= 1


def test_unmutated_definition_passes_the_pins():
    for pin in PINS:
        pin(lambda x: _definition(np.asarray(x)))
