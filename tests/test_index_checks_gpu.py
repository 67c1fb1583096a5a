"""The checked build (libgemm_f32_checked.so): device-side index checks.

Two properties, on the GPU:

* no false alarms: every kernel path that has checks (the TMA-fed pair
  kernels on whole tiles, stream-K split tiles and cluster-split tiles, the
  plain-load kernel, the SIMT kernel, the operand copy and transpose ahead of
  the pair kernels, alpha/beta, column-major storage, the allocation-free entry
  point, the host-buffer entry point in both of its forms, the reduction)
  runs through the checked build with no check failing,
  and its results still agree with the fp64 oracle;
* the checks fire: gemm_f32_selftest_index_check declares C one row short to
  the kernels, so every store to the last row fails its check and is skipped.
  The last row keeps its NaN fill, every other row agrees with the oracle, and
  the record names a C store in the last row. Every access stays inside the
  M x N matrix that was allocated, so nothing can fault.
"""

import numpy as np
import pytest

import oracle
import synth
from parity import check_within_bound, general_slack

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs(gemm_lib, checked_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return gemm_lib, checked_lib


def stream():
    return torch.cuda.current_stream().cuda_stream


def dev(x, ld=None, fill=float("nan")):
    rows, cols = x.shape
    ld = ld or cols
    buf = torch.full((rows, ld), fill, dtype=torch.float32, device="cuda")
    buf[:, :cols] = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    return buf


def take(g, cl):
    st, count, site, off, ext = g.gemm_f32_take_index_fault(stream(), lib=cl)
    assert st == g.OK, g.gemm_f32_status_string(st)
    return count, site, off, ext


def assert_clean(g, cl, what):
    st = cl.gemm_f32_poll_device_status(stream() or None)
    assert st == g.OK, f"{what}: {g.gemm_f32_status_string(st)}"
    count, site, off, ext = take(g, cl)
    assert count == 0, (f"{what}: {count} failed index checks, first at "
                        f"{g.gemm_f32_index_site_name(site)} offset {off} of {ext}")


def ex(g, cl, a, b, mode, kernel="auto", lda=None, ldb=None, ldc=None):
    m, k = a.shape
    n = b.shape[1]
    da, db = dev(a, lda), dev(b, ldb)
    ldc = ldc or n
    dc = torch.full((m, ldc), float("nan"), dtype=torch.float32, device="cuda")
    st = cl.gemm_f32_ex(m, n, k, da.data_ptr(), da.shape[1], db.data_ptr(), db.shape[1],
                        dc.data_ptr(), ldc, g.MODES[mode], g.KERNELS[kernel], stream() or None)
    assert st == g.OK, g.gemm_f32_status_string(st)
    return dc.cpu().numpy()[:, :n]


# (m, n, k, mode, kernel, lda pad, what it covers)
CASES = [
    (2048, 2048, 512, "exact", "auto", 0, "3xTF32 pair kernel, whole tiles"),
    (2048, 1280, 2048, "exact", "auto", 0, "3xTF32 pair kernel, stream-K split tiles"),
    (1024, 1024, 1024, "exact", "auto", 0, "3xTF32 pair kernel, cluster split"),
    (2048, 2048, 512, "tf32", "auto", 0, "TF32 pair kernel, whole tiles"),
    (1280, 2048, 8192, "tf32", "auto", 0, "TF32 pair kernel, stream-K split tiles"),
    (1024, 1024, 1024, "tf32", "auto", 0, "TF32 pair kernel, cluster split"),
    (1000, 1531, 777, "exact", "auto", 0, "operand copies (pitch 777) ahead of the pair kernel"),
    (300, 700, 200, "exact", "tc_lsu", 3, "plain-load kernel, 3xTF32"),
    (300, 700, 200, "tf32", "tc_lsu", 3, "plain-load kernel, one TF32 pass"),
    (257, 512, 128, "exact_simt", "auto", 0, "SIMT kernel, 16-byte copies and stores"),
    (257, 513, 129, "exact_simt", "auto", 0, "SIMT kernel, 4-byte copies and stores"),
]


@pytest.mark.parametrize("m,n,k,mode,kernel,pad,what", CASES)
def test_checked_build_no_false_alarms(libs, m, n, k, mode, kernel, pad, what):
    g, cl = libs
    take(g, cl)  # start from empty records
    a, b = synth.draw("normal", (m, k), 7 + k), synth.draw("normal", (k, n), 8 + n)
    c = ex(g, cl, a, b, mode, kernel, lda=k + pad if pad else None)
    assert_clean(g, cl, what)
    c64, s = oracle.gemm(a, b)
    check_within_bound(c, c64, s, k, mode, f"checked build: {what}")


@pytest.mark.parametrize("order,transa,transb,beta,mode", [
    (0, 1, 0, 0.0, "exact"),   # A stored K x M: transposed copy, then the pair kernel
    (0, 0, 1, 0.5, "tf32"),    # B stored N x K, beta C read by the epilogue
    (1, 0, 0, -1.0, "exact"),  # column-major storage, beta C read
    (0, 1, 1, 2.0, "exact_simt"),
])
def test_checked_build_general_forms(libs, order, transa, transb, beta, mode):
    g, cl = libs
    m, n, k = 600, 520, 384
    take(g, cl)
    a = synth.draw("uniform", (m, k), 31)
    b = synth.draw("uniform", (k, n), 32)
    c0 = synth.draw("uniform", (m, n), 33)
    alpha = 1.5
    if order == 0:
        sa, sb, sc = (a.T if transa else a), (b.T if transb else b), c0
    else:  # column-major storage of X is the row-major storage of X^T
        sa, sb, sc = (a if transa else a.T), (b if transb else b.T), c0.T
    da, db, dc = dev(sa), dev(sb), dev(sc)
    st = cl.gemm_f32_general(order, transa, transb, m, n, k, alpha, da.data_ptr(), da.shape[1],
                             db.data_ptr(), db.shape[1], beta, dc.data_ptr(), dc.shape[1],
                             g.MODES[mode], g.KERNEL_AUTO, stream() or None)
    assert st == g.OK, g.gemm_f32_status_string(st)
    assert_clean(g, cl, f"general order={order} ta={transa} tb={transb} beta={beta} {mode}")
    out = dc.cpu().numpy()
    c = out if order == 0 else out.T
    c64, s = oracle.gemm_general(a, b, alpha=alpha, beta=beta, c=c0)
    check_within_bound(c, c64, abs(alpha) * s, k, mode, "checked build, general form",
                       extra=general_slack(s, alpha, beta, c0))


def test_checked_build_noalloc(libs):
    g, cl = libs
    m, n, k = 2048, 1280, 2048  # stream-K split tiles in the fixed scratch array
    take(g, cl)
    a, b = synth.draw("normal", (m, k), 41), synth.draw("normal", (k, n), 42)
    da, db = dev(a), dev(b)
    dc = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    st = cl.gemm_f32_noalloc(m, n, k, da.data_ptr(), k, db.data_ptr(), n, dc.data_ptr(), n,
                             g.EXACT, stream() or None)
    assert st == g.OK, g.gemm_f32_status_string(st)
    assert_clean(g, cl, "allocation-free entry point")
    c64, s = oracle.gemm(a, b)
    check_within_bound(dc.cpu().numpy(), c64, s, k, "exact", "checked build, noalloc")


@pytest.mark.parametrize("mode", ["exact", "tf32"])
def test_checked_build_host_entry_point(libs, mode):
    # gemm_f32_host through the checked build: exact mode takes the fed launch
    # (ready words, done counters), tf32 mode the row chunks
    g, cl = libs
    take(g, cl)
    m, n, k = 1300, 520, 544
    a, b = synth.draw("normal", (m, k), 71), synth.draw("normal", (k, n), 72)
    ha, hb = torch.from_numpy(a).pin_memory(), torch.from_numpy(b).pin_memory()
    hc = torch.full((m, n), float("nan"), dtype=torch.float32).pin_memory()
    st = cl.gemm_f32_host(m, n, k, ha.data_ptr(), k, hb.data_ptr(), n, hc.data_ptr(), n,
                          g.MODES[mode])
    assert st == g.OK, g.gemm_f32_status_string(st)
    assert_clean(g, cl, f"host entry point, {mode}")
    c64, s = oracle.gemm(a, b)
    check_within_bound(hc.numpy(), c64, s, k, mode, f"checked build, host {mode}")


@pytest.mark.parametrize("n,offset", [((1 << 20) + 3, 0), ((1 << 20) + 5, 1), (1000, 0)])
def test_checked_build_reduction(libs, n, offset):
    g, cl = libs
    take(g, cl)
    x = synth.draw("uniform", (n + offset,), 51)
    dx = torch.from_numpy(x).cuda()
    out = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    st = cl.reduce_f32_sum(n, dx.data_ptr() + 4 * offset, out.data_ptr(), 0, stream() or None)
    assert st == g.OK, g.gemm_f32_status_string(st)
    assert_clean(g, cl, f"reduction n={n} offset={offset}")
    exact = float(np.sum(x[offset:].astype(np.float64)))
    bound = n * 2.0 ** -24 * float(np.sum(np.abs(x[offset:].astype(np.float64))))
    assert abs(float(out.item()) - exact) <= bound


# (m, n, k, mode, kernel, what)
PLANTED = [
    (2048, 2048, 512, "exact", "auto", "3xTF32 pair kernel, whole tiles"),
    (2048, 1280, 2048, "exact", "auto", "3xTF32 pair kernel, split-tile sums"),
    (1024, 1024, 1024, "exact", "auto", "3xTF32 pair kernel, cluster-split sums"),
    (2048, 2048, 512, "tf32", "auto", "TF32 pair kernel, whole tiles"),
    (300, 700, 200, "exact", "tc_lsu", "plain-load kernel"),
    (300, 260, 64, "exact_simt", "auto", "SIMT kernel, 16-byte stores"),
    (301, 257, 65, "exact_simt", "auto", "SIMT kernel, 4-byte stores"),
]


@pytest.mark.parametrize("m,n,k,mode,kernel,what", PLANTED)
def test_index_checks_fire_on_a_short_c(libs, m, n, k, mode, kernel, what):
    g, cl = libs
    take(g, cl)
    a, b = synth.draw("normal", (m, k), 61 + m), synth.draw("normal", (k, n), 62 + n)
    da, db = dev(a), dev(b)
    dc = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    st = g.gemm_f32_selftest_index_check(m, n, k, da.data_ptr(), k, db.data_ptr(), n,
                                         dc.data_ptr(), n, g.MODES[mode], g.KERNELS[kernel],
                                         stream(), lib=cl)
    assert st == g.OK, g.gemm_f32_status_string(st)
    # the status poll reports the failed checks and leaves the record in place
    assert cl.gemm_f32_poll_device_status(stream() or None) == g.ERR_INDEX
    count, site, off, ext = take(g, cl)
    assert count >= 1, what
    assert site == g.SITE_C_STORE, g.gemm_f32_index_site_name(site)
    assert ext == (m - 2) * n + n
    assert (m - 1) * n <= off < m * n, (off, what)  # an element of the last row
    # the record was reset by the read
    assert take(g, cl)[0] == 0
    assert cl.gemm_f32_poll_device_status(stream() or None) == g.OK
    c = dc.cpu().numpy()
    assert np.isnan(c[m - 1]).all(), f"{what}: a store to the last row was not skipped"
    c64, s = oracle.gemm(a, b)
    check_within_bound(c[:m - 1], c64[:m - 1], s[:m - 1], k, mode, f"short C: {what}")
