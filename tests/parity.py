"""Per-element acceptance checks shared by the parity tests.

Bounds (stated per element against the fp64 oracle, S = |A| x |B|):
  exact mode:  |C - C64| <= 2 * K * 2**-24 * S
  tf32 mode:   |C - C64| <= 2 * K * 2**-11 * S
and no NaN or Inf in C.

The tf32 bound exceeds S itself once K >= 1024, so at those sizes it would
accept any output with |C| <= S (C = 0 included). The tf32 checks therefore
also apply a bound derived from the arithmetic: each operand loses less than
2**-10 of its magnitude to the TF32 conversion, so each product is off by less
than 2**-9 of |a b|, and the fp32 accumulation adds at most K * 2**-23 * S
(allowing truncating adds):  |C - C64| <= (2**-9 + K * 2**-23) * S.
"""

import numpy as np

EXACT_MODES = ("exact", "exact_simt")


def tolerance_factor(mode: str, k: int) -> float:
    if mode in EXACT_MODES:
        return 2.0 * k * 2.0 ** -24
    if mode == "tf32":
        return 2.0 * k * 2.0 ** -11
    raise ValueError(mode)


def tf32_arithmetic_factor(k: int) -> float:
    return 2.0 ** -9 + k * 2.0 ** -23


def check_within_bound(c, c64, s, k, mode, what="", extra=0.0):
    """Element-wise acceptance of C against the oracle's C64 with scale S.

    ``extra`` (scalar or array) is added to both bounds: the rounding of a
    scale-and-add epilogue in the general form (see ``general_slack``).
    """
    c = np.asarray(c, dtype=np.float32)
    assert c.shape == c64.shape, (c.shape, c64.shape)
    finite = np.isfinite(c)
    assert finite.all(), f"{what}: {int((~finite).sum())} non-finite outputs"
    tol = tolerance_factor(mode, k) * s + extra
    err = np.abs(c.astype(np.float64) - c64)
    bad = err > tol
    if bad.any():
        idx = np.argwhere(bad)[0]
        i = tuple(int(v) for v in idx)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outputs outside the {mode} bound; "
            f"first at {i}: C={c[i]!r} C64={c64[i]!r} err={err[i]:.3e} tol={tol[i]:.3e}")
    if mode == "tf32":
        tight = tf32_arithmetic_factor(k) * s + extra
        bad = err > tight
        if bad.any():
            i = tuple(int(v) for v in np.argwhere(bad)[0])
            raise AssertionError(
                f"{what}: {int(bad.sum())} of {bad.size} outputs outside the TF32 arithmetic bound; "
                f"first at {i}: C={c[i]!r} C64={c64[i]!r} err={err[i]:.3e} tol={tight[i]:.3e}")
    # normalised error: fraction of the bound actually used
    with np.errstate(divide="ignore", invalid="ignore"):
        used = np.where(tol > 0, err / tol, 0.0)
    return float(used.max()) if used.size else 0.0


def general_slack(s, alpha, beta, c0=None):
    """Rounding allowance of C = alpha * P + beta * C0 computed in fp32 on top
    of the product P (scale S): alpha * P and beta * C0 are each rounded once
    and added once (or fused), so at most 2**-22 * (|alpha| S + |beta| |C0|)
    beyond |alpha| times the product's own bound."""
    extra = 2.0 ** -22 * abs(alpha) * s
    if beta != 0.0:
        extra = extra + 2.0 ** -22 * abs(beta) * np.abs(np.asarray(c0, dtype=np.float64))
    return extra
