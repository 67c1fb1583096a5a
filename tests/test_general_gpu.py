"""Parity of gemm_f32_general -- C = alpha * op(A) op(B) + beta * C -- against
the fp64 oracle's general form, through the C ABI.

Layouts: A and B each in plain or transposed storage (the transposed B of
"Optimizing a WebGPU Matmul Kernel using Subgroups", section 7, A likewise),
in row-major and in column-major order. Random inputs are checked within the
mode's bound scaled by |alpha| plus the rounding of the scale-and-add;
integer-valued inputs with dyadic alpha and beta must match bitwise.
"""

import numpy as np
import pytest

import oracle
import synth
from parity import check_within_bound, general_slack

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

LAYOUTS = [(0, 0), (0, 1), (1, 0), (1, 1)]  # (transa, transb)
VARIANTS = [("exact", "auto"), ("exact", "tc_tma"), ("exact", "tc_lsu"), ("exact", "simt"),
            ("tf32", "auto"), ("tf32", "tc_tma"), ("tf32", "tc_lsu"), ("exact_simt", "auto")]
SCALES = [(1.0, 0.0), (-1.5, 0.25), (0.5, 1.0)]


@pytest.fixture(scope="module")
def g(gemm_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return gemm_lib


def pad4(x):
    return -(-max(x, 1) // 4) * 4


def to_dev(x, ld, fill=float("nan")):
    rows, cols = x.shape
    buf = torch.full((max(rows, 1), ld), fill, dtype=torch.float32, device="cuda")
    if rows and cols:
        buf[:rows, :cols] = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    return buf


def stored(x, trans):
    return np.ascontiguousarray(x.T) if trans else x


def run_general(g, a, b, transa, transb, alpha, beta, c0, mode, kernel, ld_pad=0):
    """Row-major call. a, b are op(A) (M x K) and op(B) (K x N); they are handed
    over in the storage the flags say. c0 (M x N) is the previous C, or None
    (C then prefilled with NaN, which beta == 0 must never read)."""
    m, k = a.shape
    n = b.shape[1]
    a_st, b_st = stored(a, transa), stored(b, transb)
    lda = a_st.shape[1] + ld_pad
    ldb = b_st.shape[1] + ld_pad
    if kernel == "tc_tma":
        # TMA needs 16-byte row pitches; A stored transposed is first copied
        # into a workspace that has one, so its own pitch may be anything
        ldb = pad4(ldb)
        if not transa:
            lda = pad4(lda)
    lda, ldb = max(lda, 1), max(ldb, 1)
    da, db = to_dev(a_st, lda), to_dev(b_st, ldb)
    ldc = max(n, 1) + ld_pad
    if c0 is None:
        dc = torch.full((max(m, 1), ldc), float("nan"), dtype=torch.float32, device="cuda")
    else:
        dc = to_dev(c0, ldc, fill=-7.0)
    s = torch.cuda.current_stream().cuda_stream
    st = g.gemm_f32_general(g.ROW_MAJOR, transa, transb, m, n, k, alpha, da.data_ptr(), lda,
                            db.data_ptr(), ldb, beta, dc.data_ptr(), ldc, g.MODES[mode],
                            g.KERNELS[kernel], s)
    assert st == g.OK, g.gemm_f32_status_string(st)
    assert g.gemm_f32_poll_device_status(s) == g.OK
    full = dc.cpu().numpy()
    if c0 is not None and ldc > n:
        assert np.all(full[:m, n:] == -7.0), "padding of C was written"
    return full[:m, :n]


def expect(a, b, transa, transb, alpha, beta, c0, rows=None):
    return oracle.gemm_general(stored(a, transa), stored(b, transb), opa=transa, opb=transb,
                               alpha=alpha, beta=beta, c=c0, rows=rows)


@pytest.mark.parametrize("mode,kernel", VARIANTS)
@pytest.mark.parametrize("transa,transb", LAYOUTS)
@pytest.mark.parametrize("m,n,k", [(300, 700, 200), (257, 513, 129), (129, 33, 1000)])
def test_general_random_within_bound(g, mode, kernel, transa, transb, m, n, k):
    a = synth.normal((m, k), 300 + m)
    b = synth.normal((k, n), 400 + n)
    c0 = synth.normal((m, n), 500 + k)
    for alpha, beta in SCALES:
        c = run_general(g, a, b, transa, transb, alpha, beta, c0 if beta else None, mode, kernel)
        out64, s = expect(a, b, transa, transb, alpha, beta, c0)
        check_within_bound(c, out64, abs(alpha) * s, k, mode,
                           f"{mode}/{kernel} T{transa}{transb} {m}x{n}x{k} a={alpha} b={beta}",
                           extra=general_slack(s, alpha, beta, c0))


@pytest.mark.parametrize("mode,kernel", VARIANTS)
@pytest.mark.parametrize("transa,transb", LAYOUTS)
def test_general_integers_bitwise(g, mode, kernel, transa, transb):
    # small integers, dyadic scales: every kernel's result is exact
    for (m, n, k) in [(300, 700, 200), (33, 17, 48), (257, 129, 77)]:
        a = synth.small_integers((m, k), 61 + k)
        b = synth.small_integers((k, n), 62 + k)
        c0 = synth.small_integers((m, n), 63 + k)
        c = run_general(g, a, b, transa, transb, 2.0, -0.5, c0, mode, kernel, ld_pad=3)
        out64, _ = expect(a, b, transa, transb, 2.0, -0.5, c0)
        assert np.array_equal(c.astype(np.float64), out64), f"{mode}/{kernel} {m}x{n}x{k}"


@pytest.mark.parametrize("mode,kernel", [("exact", "auto"), ("tf32", "auto"), ("exact_simt", "auto"),
                                         ("exact", "tc_lsu")])
@pytest.mark.parametrize("transa,transb", LAYOUTS)
def test_general_stream_k_adds_beta_c_once(g, mode, kernel, transa, transb):
    # few output tiles and a long k range: every tile's k range is split over
    # several SMs (the TMA-fed pair kernels over the pairs of one cluster, the
    # plain-load kernel through the workspace); beta * C must enter exactly once
    m, n, k = 256, 384, 6144
    a = synth.small_integers((m, k), 71)
    b = synth.small_integers((k, n), 72)
    c0 = synth.small_integers((m, n), 73)
    c = run_general(g, a, b, transa, transb, 1.0, 1.0, c0, mode, kernel)
    out64, _ = expect(a, b, transa, transb, 1.0, 1.0, c0)
    assert np.array_equal(c.astype(np.float64), out64)


@pytest.mark.parametrize("mode", ["exact", "tf32", "exact_simt"])
def test_general_degenerate_scales(g, mode):
    m, n, k = 130, 260, 70
    a = synth.normal((m, k), 81)
    b = synth.normal((k, n), 82)
    c0 = synth.normal((m, n), 83)
    # alpha == 0: C = beta * C, A and B not used
    c = run_general(g, a, b, 0, 0, 0.0, 0.5, c0, mode, "auto")
    assert np.array_equal(c, (0.5 * c0.astype(np.float64)).astype(np.float32))
    # alpha == 0 and beta == 0: C = 0 even over NaN
    c = run_general(g, a, b, 0, 1, 0.0, 0.0, None, mode, "auto")
    assert np.all(c == 0.0)
    # K == 0: the empty product, C = beta * C
    e_a, e_b = np.zeros((m, 0), np.float32), np.zeros((0, n), np.float32)
    c = run_general(g, e_a, e_b, 0, 0, 3.0, -2.0, c0, mode, "auto")
    assert np.array_equal(c, (-2.0 * c0.astype(np.float64)).astype(np.float32))
    # beta == 0 over a NaN-filled C: nothing of the old C is read
    c = run_general(g, a, b, 1, 0, 1.0, 0.0, None, mode, "auto")
    assert np.isfinite(c).all()
    # beta == 1, alpha == 1 is accumulation
    c = run_general(g, a, b, 0, 1, 1.0, 1.0, c0, mode, "auto")
    out64, s = expect(a, b, 0, 1, 1.0, 1.0, c0)
    check_within_bound(c, out64, s, k, mode, "accumulate", extra=general_slack(s, 1.0, 1.0, c0))


@pytest.mark.parametrize("mode", ["exact", "tf32", "exact_simt"])
@pytest.mark.parametrize("transa,transb", LAYOUTS)
def test_general_column_major(g, mode, transa, transb):
    # Column-major storage: element (i, j) of a matrix with pitch ld at
    # [j * ld + i]. A column-major M x K matrix is the row-major storage of its
    # K x M transpose.
    m, n, k = 190, 75, 140
    a = synth.normal((m, k), 91)
    b = synth.normal((k, n), 92)
    c0 = synth.normal((m, n), 93)
    alpha, beta = -0.75, 0.5
    a_st = stored(a, transa)      # the stored matrix, as a logical array
    b_st = stored(b, transb)
    lda, ldb, ldc = a_st.shape[0] + 5, b_st.shape[0] + 2, m + 1
    da = to_dev(np.ascontiguousarray(a_st.T), lda)  # column-major = row-major of the transpose
    db = to_dev(np.ascontiguousarray(b_st.T), ldb)
    dc = to_dev(np.ascontiguousarray(c0.T), ldc, fill=-7.0)
    s = torch.cuda.current_stream().cuda_stream
    st = g.gemm_f32_general(g.COL_MAJOR, transa, transb, m, n, k, alpha, da.data_ptr(), lda,
                            db.data_ptr(), ldb, beta, dc.data_ptr(), ldc, g.MODES[mode],
                            g.KERNEL_AUTO, s)
    assert st == g.OK, g.gemm_f32_status_string(st)
    assert g.gemm_f32_poll_device_status(s) == g.OK
    full = dc.cpu().numpy()
    assert np.all(full[:, m:] == -7.0)
    c = full[:n, :m].T
    out64, sc = expect(a, b, transa, transb, alpha, beta, c0)
    check_within_bound(c, out64, abs(alpha) * sc, k, mode, f"col-major T{transa}{transb}",
                       extra=general_slack(sc, alpha, beta, c0))


def test_general_matches_plain_entry_point_bitwise(g):
    # gemm_f32 is the general form with alpha = 1, beta = 0, no transposes
    m, n, k = 1000, 1531, 777
    a = synth.uniform_pm1((m, k), 95)
    b = synth.uniform_pm1((k, n), 96)
    for mode in ("exact", "tf32", "exact_simt"):
        plain = torch.empty((m, n), dtype=torch.float32, device="cuda")
        da, db = to_dev(a, k), to_dev(b, n)
        s = torch.cuda.current_stream().cuda_stream
        assert g.gemm_f32(m, n, k, da.data_ptr(), k, db.data_ptr(), n, plain.data_ptr(), n,
                          g.MODES[mode], s) == g.OK
        gen = run_general(g, a, b, 0, 0, 1.0, 0.0, None, mode, "auto")
        assert np.array_equal(plain.cpu().numpy(), gen), mode


# The product A B of the 4096^3 operands, computed once by the oracle: every
# storage of A and B below holds the same two matrices.
_FULL = {}


def _full_product(a, b):
    if "ab" not in _FULL:
        _FULL["ab"] = oracle.gemm(a, b)
    return _FULL["ab"]


@pytest.mark.slow
@pytest.mark.parametrize("mode", ["exact", "tf32"])
@pytest.mark.parametrize("transa,transb", LAYOUTS)
def test_general_full_size(g, mode, transa, transb):
    # 4096^3 in the launch configuration of the benchmark (TMA-fed kernel when
    # the layout allows it): every element against alpha * (A B) + beta * C0
    # from the oracle's product, and sampled rows against the oracle's general
    # form applied to the operands as stored
    m = n = k = 4096
    a = synth.uniform_pm1((m, k), 1008)
    b = synth.uniform_pm1((k, n), 1009)
    c0 = synth.uniform_pm1((m, n), 1010)
    alpha, beta = 1.25, -0.5
    c = run_general(g, a, b, transa, transb, alpha, beta, c0, mode, "auto")
    c64, s = _full_product(a, b)
    full64 = alpha * c64 + beta * c0.astype(np.float64)
    check_within_bound(c, full64, abs(alpha) * s, k, mode, f"4096^3 T{transa}{transb} full",
                       extra=general_slack(s, alpha, beta, c0))
    rows = np.array([0, 1, 255, 256, 2047, 3000, 4095])
    out64, s_rows = expect(a, b, transa, transb, alpha, beta, c0, rows=rows)
    check_within_bound(c[rows], out64, abs(alpha) * s_rows, k, mode, f"4096^3 T{transa}{transb}",
                       extra=general_slack(s_rows, alpha, beta, c0[rows]))


@pytest.mark.slow
@pytest.mark.parametrize("mode", ["exact", "tf32"])
def test_general_full_size_reruns_bitwise(g, mode):
    # alpha * A B + beta * C at 4096^3, five calls on the same inputs: the
    # scaled epilogue computes alpha * acc from registers that a TMEM load
    # fills asynchronously, so a use scheduled before the load's wait would
    # read stale values in some calls and not others. Every call must give
    # the same bits, and the first must meet the bound against the oracle.
    m = n = k = 4096
    a = synth.uniform_pm1((m, k), 1008)
    b = synth.uniform_pm1((k, n), 1009)
    c0 = synth.uniform_pm1((m, n), 1010)
    alpha, beta = 1.25, -0.5
    first = run_general(g, a, b, 0, 0, alpha, beta, c0, mode, "auto")
    for _ in range(4):
        c = run_general(g, a, b, 0, 0, alpha, beta, c0, mode, "auto")
        assert np.array_equal(c.view(np.uint32), first.view(np.uint32)), \
            f"{mode}: {int((c != first).sum())} outputs differ between calls"
    c64, s = _full_product(a, b)
    full64 = alpha * c64 + beta * c0.astype(np.float64)
    check_within_bound(first, full64, abs(alpha) * s, k, mode, "4096^3 reruns",
                       extra=general_slack(s, alpha, beta, c0))
