"""Pins for the fp64 oracle (CPU only).

The oracle must be right before it can vouch for the CUDA path, so it is checked
here against things other than itself: hand-worked products, algebraic
structure (identity, permutation, diagonal, transpose, linearity, scaling),
the all-ones closed form, exact rational brute force, the integer-valued
self-test pattern of "GPU compute shaders" (section "Code"), and strided
layouts. ``test_pins_catch_planted_mistakes`` shows that a plausible slip in
the oracle (a transposed operand, a dropped term, a wrong sign, an index
off by one) fails at least one of these pins.
"""

import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    mats = {}
    with open(os.path.join(GOLDEN, name)) as f:
        lines = [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]
    it = iter(lines)
    for ln in it:
        tag, r, c = ln.split()
        r, c = int(r), int(c)
        mats[tag] = np.array([[float(v) for v in next(it).split()] for _ in range(r)]).reshape(r, c)
    return mats


GOLDEN_FILES = sorted(f for f in os.listdir(GOLDEN) if f.startswith("hand_"))


# --- the pins, written so that they can also be run against a mutant --------

def pin_golden(gemm):
    for name in GOLDEN_FILES:
        g = _read_golden(name)
        c64, s = gemm(g["A"].astype(np.float32), g["B"].astype(np.float32))
        if not (np.array_equal(c64, g["C"]) and np.array_equal(s, g["S"])):
            return f"golden {name}"
    return None


def pin_structure(gemm):
    rng = np.random.default_rng(7)
    for m, n, k in [(5, 7, 3), (16, 9, 16), (1, 1, 1), (33, 17, 12)]:
        a = synth.uniform_pm1((m, k), 11 + m)
        b = synth.uniform_pm1((k, n), 12 + n)
        # A x I = A and I x B = B, exactly
        if not np.array_equal(gemm(a, np.eye(k, dtype=np.float32))[0], a.astype(np.float64)):
            return "right identity"
        if not np.array_equal(gemm(np.eye(k, dtype=np.float32), b)[0], b.astype(np.float64)):
            return "left identity"
        # P x B permutes the rows of B
        perm = rng.permutation(k)
        p = np.zeros((k, k), dtype=np.float32)
        p[np.arange(k), perm] = 1.0
        if not np.array_equal(gemm(p, b)[0], b[perm].astype(np.float64)):
            return "row permutation"
        # B x P permutes the columns of B (P now n x n)
        permn = rng.permutation(n)
        pn = np.zeros((n, n), dtype=np.float32)
        pn[permn, np.arange(n)] = 1.0
        if not np.array_equal(gemm(b, pn)[0], b[:, permn].astype(np.float64)):
            return "column permutation"
        # D x B scales the rows of B (products of two fp32 values are exact in fp64)
        d = synth.uniform_pm1((k,), 99 + k)
        got = gemm(np.diag(d).astype(np.float32), b)[0]
        if not np.array_equal(got, d.astype(np.float64)[:, None] * b.astype(np.float64)):
            return "diagonal scaling"
        # (A B)^T = B^T A^T: same products, same k order, so bitwise equal
        c = gemm(a, b)[0]
        ct = gemm(np.ascontiguousarray(b.T), np.ascontiguousarray(a.T))[0]
        if not np.array_equal(c.T, ct):
            return "transpose identity"
        # scaling A by 2 scales C by 2 exactly
        if not np.array_equal(gemm((2 * a).astype(np.float32), b)[0], 2 * c):
            return "scaling"
    return None


def pin_all_ones(gemm):
    for m, n, k in [(1, 1, 1), (3, 5, 7), (17, 1, 129), (128, 129, 257), (2, 3, 4096)]:
        c64, s = gemm(np.ones((m, k), np.float32), np.ones((k, n), np.float32))
        if not (np.all(c64 == k) and np.all(s == k)):
            return f"all-ones {m}x{n}x{k}"
    return None


def pin_linearity(gemm):
    # B1 and B2 carry at most 12 significant bits, so B1 + B2 is exact in fp32
    for m, n, k in [(7, 9, 13), (32, 24, 16)]:
        a = synth.uniform_pm1((m, k), 21)
        b1 = np.round(synth.uniform_pm1((k, n), 22) * 2048) / 2048
        b2 = np.round(synth.uniform_pm1((k, n), 23) * 2048) / 2048
        b1, b2 = b1.astype(np.float32), b2.astype(np.float32)
        lhs, s = gemm(a, (b1 + b2).astype(np.float32))
        r1, s1 = gemm(a, b1)
        r2, s2 = gemm(a, b2)
        # exact up to fp64 accumulation rounding (K * 2^-52 relative to the scales)
        tol = 4 * k * 2.0 ** -52 * (s + s1 + s2)
        if not np.all(np.abs(lhs - (r1 + r2)) <= tol):
            return "linearity"
    return None


def pin_brute_force(gemm):
    # exact rational arithmetic on tiny random inputs
    for trial, (m, n, k) in enumerate([(1, 1, 1), (2, 3, 5), (4, 4, 4), (3, 6, 9), (5, 2, 17)]):
        a = synth.normal((m, k), 300 + trial)
        b = synth.normal((k, n), 400 + trial)
        c64, s = gemm(a, b)
        for i in range(m):
            for j in range(n):
                exact = sum(Fraction(float(a[i, kk])) * Fraction(float(b[kk, j])) for kk in range(k))
                scale = sum(abs(Fraction(float(a[i, kk])) * Fraction(float(b[kk, j]))) for kk in range(k))
                if abs(Fraction(c64[i, j]) - exact) > Fraction(k) * Fraction(2) ** -52 * scale:
                    return "brute force value"
                if abs(Fraction(s[i, j]) - scale) > Fraction(k) * Fraction(2) ** -52 * scale:
                    return "brute force scale"
    return None


def pin_integer_selftest(gemm):
    # the integer-valued pattern of "GPU compute shaders" (section "Code"):
    # A[i] = (i mod 7) - 3 over m x k, B[i] = (i mod 5) - 2 over k x n, m, n, k = 32, 24, 16;
    # all values are small integers, so the result is exact
    m, n, k = 32, 24, 16
    # element (row, col) of each operand takes the pattern at its row-major
    # linear index
    a_int = [[(row * k + col) % 7 - 3 for col in range(k)] for row in range(m)]
    b_int = [[(row * n + col) % 5 - 2 for col in range(n)] for row in range(k)]
    c64, _ = gemm(np.array(a_int, dtype=np.float32), np.array(b_int, dtype=np.float32))
    # the product in Python integers (exact)
    b_cols = list(zip(*b_int))
    want = [[sum(x * y for x, y in zip(a_row, b_col)) for b_col in b_cols] for a_row in a_int]
    if not np.array_equal(c64, np.array(want, dtype=np.float64)):
        return "integer self-test"
    return None


ALL_PINS = [pin_golden, pin_structure, pin_all_ones, pin_linearity, pin_brute_force,
            pin_integer_selftest]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    assert pin(oracle.gemm) is None


def test_pins_catch_planted_mistakes():
    """Each planted slip in the oracle's arithmetic fails at least one pin."""

    def transposed_b(a, b):          # reads B as if it were stored transposed
        if b.shape[0] == b.shape[1]:
            return oracle.gemm(a, np.ascontiguousarray(b.T))
        return oracle.gemm(a, b)  # shape mismatch would raise; only square B mutates

    def dropped_last_term(a, b):     # k loop stops one short
        if a.shape[1] <= 1:
            return oracle.gemm(a, b)
        return oracle.gemm(np.ascontiguousarray(a[:, :-1]), np.ascontiguousarray(b[:-1]))

    def wrong_sign(a, b):            # one product subtracted instead of added
        c, s = oracle.gemm(a, b)
        a0 = a[:, :1].astype(np.float64)
        b0 = b[:1, :].astype(np.float64)
        return c - 2 * a0 * b0, s

    def row_off_by_one(a, b):        # reads row i+1 of A (wrapping)
        return oracle.gemm(np.ascontiguousarray(np.roll(a, -1, axis=0)), b)

    def scale_without_abs(a, b):     # S computed without absolute values
        c, _ = oracle.gemm(a, b)
        return c, c

    for mutant in (transposed_b, dropped_last_term, wrong_sign, row_off_by_one, scale_without_abs):
        failed = [p.__name__ for p in ALL_PINS if p(mutant) is not None]
        assert failed, f"no pin catches the planted mistake {mutant.__name__}"


@pytest.mark.parametrize("m,n,k", [(1, 1, 1), (7, 5, 3), (33, 65, 17), (128, 96, 40)])
def test_rows_and_entries_agree_with_full(m, n, k):
    a = synth.normal((m, k), 5)
    b = synth.normal((k, n), 6)
    c64, s = oracle.gemm(a, b)
    rows = np.unique(np.array([0, m - 1, m // 2, m // 3]))
    cr, sr = oracle.gemm_rows(a, b, rows)
    assert np.array_equal(cr, c64[rows]) and np.array_equal(sr, s[rows])
    rng = np.random.default_rng(0)
    ii = rng.integers(0, m, 50)
    jj = rng.integers(0, n, 50)
    ce, se = oracle.gemm_entries(a, b, ii, jj)
    assert np.array_equal(ce, c64[ii, jj]) and np.array_equal(se, s[ii, jj])


def test_strided_operands_match_dense():
    m, n, k = 19, 23, 29
    a = synth.uniform_pm1((m, k), 1)
    b = synth.uniform_pm1((k, n), 2)
    ref = oracle.gemm(a, b)
    a_pad = synth.embed_strided(a, 37)[:, :k]
    b_pad = synth.embed_strided(b, 31)[:, :n]
    got = oracle.gemm(a_pad, b_pad)
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


def test_agrees_with_library_fp64_matmul():
    # numpy's fp64 matmul is a different summation order; both are within
    # fp64 rounding of the exact value
    for m, n, k in [(64, 48, 300), (5, 130, 777)]:
        a = synth.normal((m, k), 8)
        b = synth.normal((k, n), 9)
        c64, s = oracle.gemm(a, b)
        ref = a.astype(np.float64) @ b.astype(np.float64)
        assert np.all(np.abs(c64 - ref) <= 2 * k * 2.0 ** -53 * s)


def test_empty_and_degenerate_shapes():
    # K == 0: the empty sum is zero
    c64, s = oracle.gemm(np.zeros((3, 0), np.float32), np.zeros((0, 4), np.float32))
    assert c64.shape == (3, 4) and not c64.any() and not s.any()
    # M == 0 or N == 0: empty output
    assert oracle.gemm(np.zeros((0, 5), np.float32), np.zeros((5, 4), np.float32))[0].shape == (0, 4)
    assert oracle.gemm(np.zeros((3, 5), np.float32), np.zeros((5, 0), np.float32))[0].shape == (3, 0)


def test_input_generators_are_deterministic_and_in_range():
    u = synth.uniform_pm1((1000,), 1234)
    assert np.array_equal(u, synth.uniform_pm1((1000,), 1234))
    assert u.min() >= -1.0 and u.max() < 1.0
    assert np.all(u * 2 ** 23 == np.round(u * 2 ** 23))  # on the 2^-23 grid, exact in fp32
    assert not np.array_equal(u, synth.uniform_pm1((1000,), 1235))
    z = synth.normal((100000,), 77)
    assert abs(float(z.mean())) < 0.02 and abs(float(z.std()) - 1) < 0.02
    i = synth.small_integers((1000,), 5)
    assert i.min() >= -8 and i.max() <= 8 and np.all(i == np.round(i))
    # known SplitMix64 outputs: the first three values of the reference
    # generator seeded with 0 (state advanced by the golden gamma before mixing)
    v = synth.splitmix64(0, np.arange(3, dtype=np.uint64))
    assert [int(x) for x in v] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_num_threads_reported():
    assert oracle.num_threads() >= 1


# --- the general form: alpha * A op(B) + beta * C -----------------------------

@pytest.mark.parametrize("m,n,k", [(1, 1, 1), (7, 5, 3), (33, 65, 17)])
def test_general_reduces_to_the_plain_product(m, n, k):
    a = synth.normal((m, k), 51)
    b = synth.normal((k, n), 52)
    c64, s = oracle.gemm(a, b)
    g64, gs = oracle.gemm_general(a, b)
    assert np.array_equal(g64, c64) and np.array_equal(gs, s)
    # B supplied transposed: same products, same k order, so bitwise equal
    t64, ts = oracle.gemm_general(a, np.ascontiguousarray(b.T), opb=1)
    assert np.array_equal(t64, c64) and np.array_equal(ts, s)
    # A supplied transposed (K x M), and both
    t64, ts = oracle.gemm_general(np.ascontiguousarray(a.T), b, opa=1)
    assert np.array_equal(t64, c64) and np.array_equal(ts, s)
    t64, ts = oracle.gemm_general(np.ascontiguousarray(a.T), np.ascontiguousarray(b.T), opa=1,
                                  opb=1)
    assert np.array_equal(t64, c64) and np.array_equal(ts, s)


@pytest.mark.parametrize("name", ["hand_2x2.txt", "hand_3x2x4.txt"])
@pytest.mark.parametrize("opa,opb", [(0, 1), (1, 0), (1, 1)])
def test_general_transposed_storage_hand_worked(name, opa, opb):
    # The hand-worked fixtures, with the operands handed over in transposed
    # storage (the transposed B of the subgroups page, section 7; A likewise).
    g = _read_golden(name)
    a = g["A"].astype(np.float32)
    b = g["B"].astype(np.float32)
    a_st = np.ascontiguousarray(a.T) if opa else a
    b_st = np.ascontiguousarray(b.T) if opb else b
    out, s = oracle.gemm_general(a_st, b_st, opa=opa, opb=opb)
    assert np.array_equal(out, g["C"])
    assert np.array_equal(s, g["S"])


def test_general_scaling_and_accumulation():
    m, n, k = 9, 11, 13
    a = synth.small_integers((m, k), 53)
    b = synth.small_integers((k, n), 54)
    c = synth.small_integers((m, n), 55)
    c64, _ = oracle.gemm(a, b)
    # exact for small integers and dyadic scales
    out, _ = oracle.gemm_general(a, b, alpha=2.0, beta=-0.5, c=c)
    assert np.array_equal(out, 2.0 * c64 - 0.5 * c.astype(np.float64))
    out, _ = oracle.gemm_general(a, b, alpha=0.0, beta=1.0, c=c)
    assert np.array_equal(out, c.astype(np.float64))
    # beta == 0 never reads C (NaN there does not propagate)
    nanc = np.full((m, n), np.nan, np.float32)
    out, _ = oracle.gemm_general(a, b, alpha=1.0, beta=0.0, c=nanc)
    assert np.array_equal(out, c64)
    # hand-worked: the 2x2 fixture with alpha = 1, beta = 1, C = [[1, 1], [1, 1]]
    g = _read_golden("hand_2x2.txt")
    out, _ = oracle.gemm_general(g["A"].astype(np.float32), g["B"].astype(np.float32), alpha=1.0,
                                 beta=1.0, c=np.ones((2, 2), np.float32))
    assert np.array_equal(out, g["C"] + 1)


def test_general_rows_select():
    a = synth.normal((20, 7), 56)
    b = synth.normal((7, 9), 57)
    full, s = oracle.gemm_general(a, b)
    part, ps = oracle.gemm_general(a, b, rows=[19, 0, 5])
    assert np.array_equal(part, full[[19, 0, 5]]) and np.array_equal(ps, s[[19, 0, 5]])
