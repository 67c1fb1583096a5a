"""Parity of the CUDA path (through the C ABI) against the fp64 oracle.

Every comparison is element by element: within the mode's bound for random
inputs, bitwise for integer-valued inputs (where every kernel's result is
exact). Inputs come from ``synth``; expected values only from ``oracle``.
"""

import numpy as np
import pytest

import oracle
import synth
from parity import check_within_bound

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

MODES = ["exact", "tf32", "exact_simt"]
# (mode, kernel) pairs that are legal for TMA-legal operands
VARIANTS = [("exact", "auto"), ("exact", "tc_tma"), ("exact", "tc_lsu"), ("exact", "simt"),
            ("tf32", "tc_tma"), ("tf32", "tc_lsu"), ("exact_simt", "auto")]


@pytest.fixture(scope="module")
def g(gemm_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return gemm_lib


def to_dev(x, ld=None, fill=float("nan")):
    """Upload a rows x cols fp32 matrix into a (rows x ld) device buffer."""
    rows, cols = x.shape
    ld = ld or max(cols, 1)
    buf = torch.full((max(rows, 1), ld), fill, dtype=torch.float32, device="cuda")
    if rows and cols:
        buf[:rows, :cols] = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    return buf


def run(g, a, b, mode="exact", kernel="auto", lda=None, ldb=None, ldc=None, c_fill=float("nan")):
    """C = A x B through gemm_f32_ex; returns (C as numpy, full C buffer as numpy)."""
    m, k = a.shape
    _, n = b.shape
    if kernel == "tc_tma":
        # the TMA-fed kernel needs row pitches that are multiples of 16 bytes
        lda = lda or -(-max(k, 1) // 4) * 4
        ldb = ldb or -(-max(n, 1) // 4) * 4
    da, db = to_dev(a, lda), to_dev(b, ldb)
    ldc = ldc or max(n, 1)
    dc = torch.full((max(m, 1), ldc), c_fill, dtype=torch.float32, device="cuda")
    st = g.gemm_f32_ex(m, n, k, da.data_ptr(), da.shape[1], db.data_ptr(), db.shape[1],
                       dc.data_ptr(), ldc, g.MODES[mode], g.KERNELS[kernel],
                       torch.cuda.current_stream().cuda_stream)
    assert st == g.OK, g.gemm_f32_status_string(st)
    assert g.gemm_f32_poll_device_status(torch.cuda.current_stream().cuda_stream) == g.OK
    full = dc.cpu().numpy()
    return full[:m, :n], full


_CONFIG_CACHE = {}


def config_operands(name):
    if name not in _CONFIG_CACHE:
        _CONFIG_CACHE.clear()  # keep at most one full-size workload in host memory
        _CONFIG_CACHE[name] = synth.config_operands(name)
    return _CONFIG_CACHE[name]


def operands(m, n, k, dist="uniform", seed=0):
    return (synth.draw(dist, (m, k), 100 + seed), synth.draw(dist, (k, n), 200 + seed))


@pytest.mark.parametrize("mode,kernel", VARIANTS)
@pytest.mark.parametrize("m,n,k", [(300, 700, 200), (257, 513, 129), (128, 256, 32),
                                   (1, 1, 64), (129, 33, 1000)])
def test_random_within_bound(g, mode, kernel, m, n, k):
    a, b = operands(m, n, k, "normal", seed=m + n + k)
    c, _ = run(g, a, b, mode, kernel)
    c64, s = oracle.gemm(a, b)
    check_within_bound(c, c64, s, k, mode, f"{mode}/{kernel} {m}x{n}x{k}")


@pytest.mark.parametrize("mode,kernel", VARIANTS)
def test_integer_inputs_bitwise(g, mode, kernel):
    # small integers: every kernel's result is exact, so it equals the oracle bitwise
    for (m, n, k) in [(300, 700, 200), (32, 24, 16), (257, 129, 77)]:
        a = synth.small_integers((m, k), 31 + k)
        b = synth.small_integers((k, n), 32 + k)
        c, _ = run(g, a, b, mode, kernel)
        c64, _ = oracle.gemm(a, b)
        assert np.array_equal(c.astype(np.float64), c64), f"{mode}/{kernel} {m}x{n}x{k}"


@pytest.mark.parametrize("mode,kernel", [("exact", "tc_tma"), ("tf32", "tc_tma"), ("exact", "simt")])
def test_integer_selftest_pattern(g, mode, kernel):
    # the integer pattern of "GPU compute shaders" (section "Code"), m, n, k = 32, 24, 16
    m, n, k = 32, 24, 16
    a = (np.arange(m * k) % 7 - 3).astype(np.float32).reshape(m, k)
    b = (np.arange(k * n) % 5 - 2).astype(np.float32).reshape(k, n)
    c, _ = run(g, a, b, mode, kernel)
    assert np.array_equal(c.astype(np.float64), oracle.gemm(a, b)[0])


@pytest.mark.parametrize("mode,kernel", VARIANTS)
def test_all_ones_closed_form(g, mode, kernel):
    for (m, n, k) in [(1, 1, 1), (129, 257, 33), (200, 300, 1000)]:
        c, _ = run(g, np.ones((m, k), np.float32), np.ones((k, n), np.float32), mode, kernel)
        assert np.all(c == k), f"{mode}/{kernel} {m}x{n}x{k}"


@pytest.mark.parametrize("mode,kernel", [("exact", "tc_lsu"), ("tf32", "tc_lsu"), ("exact", "simt"),
                                         ("exact", "auto"), ("tf32", "auto"), ("exact", "tc_tma"),
                                         ("tf32", "tc_tma")])
def test_ragged_strides_and_guard_bands(g, mode, kernel):
    # odd leading dimensions (TMA cannot read them: the TMA-fed kernel works on
    # copies with 16-byte pitches), NaN padding in A and B, sentinel padding in
    # C: padding must never be read into a result or written
    m, n, k = 203, 301, 117
    a, b = operands(m, n, k, "normal", seed=5)
    c, full = run(g, a, b, mode, kernel, lda=k + 3, ldb=n + 5, ldc=n + 7, c_fill=-12345.0)
    c64, s = oracle.gemm(a, b)
    check_within_bound(c, c64, s, k, mode, f"ragged {mode}/{kernel}")
    assert np.all(full[:, n:] == -12345.0), "write outside C's columns"


@pytest.mark.parametrize("mode,kernel", [("exact", "auto"), ("tf32", "auto"), ("exact", "tc_lsu")])
@pytest.mark.parametrize("off_a,off_b", [(1, 0), (0, 3), (2, 1)])
def test_misaligned_bases(g, mode, kernel, off_a, off_b):
    # A and B starting 4, 8 or 12 bytes past a 16-byte boundary, NaN before
    # and after them: TMA cannot read them in place, so they are copied
    m, n, k = 300, 260, 190
    a, b = operands(m, n, k, "normal", seed=off_a * 4 + off_b)
    ba = torch.full((m * k + 8,), float("nan"), device="cuda")
    bb = torch.full((k * n + 8,), float("nan"), device="cuda")
    ba[off_a:off_a + m * k] = torch.from_numpy(a.reshape(-1)).cuda()
    bb[off_b:off_b + k * n] = torch.from_numpy(b.reshape(-1)).cuda()
    dc = torch.full((m, n), float("nan"), device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = g.gemm_f32_ex(m, n, k, ba.data_ptr() + 4 * off_a, k, bb.data_ptr() + 4 * off_b, n,
                       dc.data_ptr(), n, g.MODES[mode], g.KERNELS[kernel], s)
    assert st == g.OK, g.gemm_f32_status_string(st)
    assert g.gemm_f32_poll_device_status(s) == g.OK
    c64, sc = oracle.gemm(a, b)
    check_within_bound(dc.cpu().numpy(), c64, sc, k, mode, f"offsets {off_a},{off_b}")


def test_ragged_sweep(g):
    # brute-force sweep of small shapes around tile edges, every kernel
    sizes = [1, 2, 3, 7, 8, 9, 15, 16, 17, 31, 32, 33, 127, 128, 129, 255, 256, 257]
    rng = np.random.default_rng(2024)
    combos = {(int(rng.choice(sizes)), int(rng.choice(sizes)), int(rng.choice(sizes)))
              for _ in range(60)}
    combos |= {(1, 1, 1), (257, 257, 257), (1, 257, 17), (257, 1, 129), (17, 17, 17)}
    for (m, n, k) in sorted(combos):
        a = synth.small_integers((m, k), m * 7 + k)
        b = synth.small_integers((k, n), n * 11 + k)
        c64, _ = oracle.gemm(a, b)
        ar, br = operands(m, n, k, "uniform", seed=m * n + k)
        r64, rs = oracle.gemm(ar, br)
        for mode, kernel in VARIANTS:
            c, _ = run(g, a, b, mode, kernel)
            assert np.array_equal(c.astype(np.float64), c64), f"int {mode}/{kernel} {m}x{n}x{k}"
            if mode == "exact" and kernel in ("tc_tma", "tc_lsu") and k < 8:
                continue  # 3xTF32 is outside the FP32 bound for K < 8 on random data
            if mode == "tf32" and k < 4:
                continue  # truncated TF32 operands: the bound needs K >= 2 (worst case)
            c, _ = run(g, ar, br, mode, kernel)
            check_within_bound(c, r64, rs, k, mode, f"rand {mode}/{kernel} {m}x{n}x{k}")


@pytest.mark.parametrize("mode,kernel", [("exact", "tc_tma"), ("tf32", "tc_tma"), ("exact", "tc_lsu"),
                                         ("tf32", "tc_lsu")])
@pytest.mark.parametrize("m,n,k", [
    (256, 128, 4096),     # one tile, k split over the most CTAs
    (200, 100, 2000),     # one ragged tile, split
    (3328, 1536, 512),    # 78 pair tiles: a full wave, the last 2 dealt whole (3xTF32: too
                          # short to split)
    (3328, 1536, 1024),   # 78 pair tiles: a full wave whole, 2 tiles split (3xTF32)
    (3328, 1536, 4096),   # a full wave of pair tiles whole, 2 tiles split
    (512, 512, 512),      # 4 pair tiles, whole (3xTF32: too short to split)
    (512, 512, 1024),     # 4 pair tiles, each split (3xTF32)
    (200, 100, 8000),     # one ragged tile, split in both modes
    (512, 512, 4096),     # 8 tiles, each split in both modes
    (2048, 1280, 2048),   # 40 pair tiles on 76 pairs: every tile split through the
                          # workspace (3xTF32; tf32: dealt whole)
    (1280, 2048, 8192),   # 40 pair tiles, split in both modes
])
def test_stream_k_splits(g, mode, kernel, m, n, k):
    # tiles whose k range is shared by several CTAs: partial sums through the
    # workspace, summed by the last contributor in part order (the TMA-fed
    # pair kernels split tiles inside a cluster instead when there are at most
    # half as many tiles as pairs, which the small shapes here exercise)
    a, b = operands(m, n, k, "normal", seed=m + 3 * n + k)
    c, _ = run(g, a, b, mode, kernel)
    rows = np.unique(np.concatenate([np.arange(0, m, max(1, m // 97)), [m - 1]]))
    c64, s = oracle.gemm_rows(a, b, rows)
    check_within_bound(c[rows], c64, s, k, mode, f"stream-K {mode}/{kernel} {m}x{n}x{k}")
    ai = synth.small_integers((m, k), 7)
    bi = synth.small_integers((k, n), 8)
    ci, _ = run(g, ai, bi, mode, kernel)
    ci64, _ = oracle.gemm_rows(ai, bi, rows)
    assert np.array_equal(ci[rows].astype(np.float64), ci64)
    c2, _ = run(g, a, b, mode, kernel)
    assert np.array_equal(c.view(np.uint32), c2.view(np.uint32)), "split tiles not deterministic"


@pytest.mark.parametrize("mode,m,n,k", [
    ("exact", 512, 512, 512),     # 4 tiles, 4 pairs per tile
    ("exact", 1000, 1531, 776),   # 24 ragged tiles, 3 pairs per tile: clusters of 6
    ("exact", 129, 257, 520),     # 2 ragged tiles, k not a multiple of the k-block
    ("exact", 300, 700, 2000),    # 6 ragged tiles, k slices of unequal length
    ("tf32", 300, 700, 2000),
    ("exact", 1024, 1024, 1024),  # 16 tiles (4 pairs per tile if 16 clusters of 8 fit)
    ("tf32", 1024, 1024, 1024),
    ("tf32", 700, 300, 1100),     # 6 ragged tiles, ragged k
    ("exact", 256, 128, 4096),    # one tile
    ("tf32", 256, 128, 4096),
])
def test_cluster_split(g, mode, m, n, k):
    # few unit tiles: pairs of one cluster take k-slices of a tile; after a
    # cluster barrier each CTA sums its band of rows over the slices, in pair
    # order (its own slice from shared memory, the others' through L2)
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    st, stats = g.gemm_f32_schedule_check(m, n, k, sms // 2, mode + "_pair")
    assert st == g.OK and stats["cluster_split"] >= 2, stats
    a, b = operands(m, n, k, "normal", seed=m + 7 * n + k)
    c, full = run(g, a, b, mode, "tc_tma", ldc=n + 3, c_fill=-777.0)
    c64, sc = oracle.gemm(a, b)
    check_within_bound(c, c64, sc, k, mode, f"cluster split {mode} {m}x{n}x{k}")
    assert np.all(full[:, n:] == -777.0), "write outside C's columns"
    c2, _ = run(g, a, b, mode, "tc_tma", ldc=n + 3)
    assert np.array_equal(c.view(np.uint32), c2.view(np.uint32)), "cluster split not deterministic"
    ai = synth.small_integers((m, k), 17)
    bi = synth.small_integers((k, n), 18)
    ci, _ = run(g, ai, bi, mode, "tc_tma")
    assert np.array_equal(ci.astype(np.float64), oracle.gemm(ai, bi)[0])


@pytest.mark.parametrize("mode", ["exact", "tf32"])
@pytest.mark.parametrize("m,n,k", [
    (256, 256, 65536),   # one pair tile, k sliced over a cluster: 512 k-blocks per slice
    (1024, 768, 40000),  # 12 tiles, cluster split, ragged k (40000 = 1250 k-blocks)
    (4096, 2560, 12288), # 160 tiles: two whole waves, the rest stream-K parts
])
def test_long_k(g, mode, m, n, k):
    # many k-blocks accumulated per tile, in one accumulator and across the
    # parts of split tiles. Integer inputs in [-8, 8] keep every partial sum an
    # integer below 2^24 (|sum| <= 64 K), exact in fp32 and TF32 alike, so the
    # sampled rows must equal the fp64 oracle bit for bit; random inputs must
    # stay within the mode's bound.
    rows = np.unique(np.concatenate([np.arange(0, m, max(1, m // 23)), [m - 1]]))
    ai = synth.small_integers((m, k), 21 + k)
    bi = synth.small_integers((k, n), 22 + k)
    ci, _ = run(g, ai, bi, mode, "auto")
    ci64, _ = oracle.gemm_rows(ai, bi, rows)
    assert np.array_equal(ci[rows].astype(np.float64), ci64), f"long k {mode} {m}x{n}x{k}"
    a, b = operands(m, n, k, "uniform", seed=k + n)
    c, _ = run(g, a, b, mode, "auto")
    c64, s = oracle.gemm_rows(a, b, rows)
    check_within_bound(c[rows], c64, s, k, mode, f"long k {mode} {m}x{n}x{k}")


def test_nan_prefilled_output_fully_written(g):
    for mode, kernel in VARIANTS:
        a, b = operands(385, 519, 96, "uniform", seed=9)
        c, _ = run(g, a, b, mode, kernel, c_fill=float("nan"))
        assert np.isfinite(c).all(), f"{mode}/{kernel} left outputs unwritten"


def test_rerun_is_bitwise_identical(g):
    a, b = operands(640, 768, 512, "normal", seed=3)
    for mode, kernel in VARIANTS:
        c1, _ = run(g, a, b, mode, kernel)
        c2, _ = run(g, a, b, mode, kernel)
        assert np.array_equal(c1.view(np.uint32), c2.view(np.uint32)), f"{mode}/{kernel}"


def test_k_zero_writes_zeros_and_empty_is_noop(g):
    for mode in MODES:
        c, _ = run(g, np.zeros((5, 0), np.float32), np.zeros((0, 7), np.float32), mode, c_fill=3.0)
        assert np.all(c == 0.0)
    # M == 0: C untouched
    dc = torch.full((4, 4), 7.0, device="cuda")
    st = g.gemm_f32(0, 4, 4, 0, 4, 0, 4, dc.data_ptr(), 4, g.EXACT, 0)
    torch.cuda.synchronize()
    assert st == g.OK and torch.all(dc == 7.0)


def test_alias_error_on_device(g):
    x = torch.zeros((64, 64), device="cuda")
    assert g.gemm_f32(64, 64, 64, x.data_ptr(), 64, x.data_ptr(), 64, x.data_ptr(), 64,
                      g.EXACT, 0) == g.ERR_ALIAS


def test_torch_wrapper_and_streams(g):
    a, b = operands(256, 384, 128, "uniform", seed=1)
    s = torch.cuda.Stream()
    ta, tb = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    with torch.cuda.stream(s):
        out = g.matmul(ta, tb, "exact")
    s.synchronize()
    c64, sc = oracle.gemm(a, b)
    check_within_bound(out.cpu().numpy(), c64, sc, 128, "exact", "matmul on a side stream")


def test_host_entry_point(g):
    for (m, n, k), mode in [((1000, 1531, 777), "exact"), ((1000, 1531, 777), "tf32"),
                            ((64, 96, 5), "exact"), ((3, 5, 0), "tf32")]:
        a, b = operands(m, n, k, "normal", seed=k)
        c = g.matmul_host(a, b, mode)
        c64, s = oracle.gemm(a, b)
        check_within_bound(c, c64, s, k, mode, f"host {mode} {m}x{n}x{k}")


def test_host_entry_point_row_chunks(g):
    # the host entry pipelines row chunks of A and C through two copy streams
    # (1024-row chunks and up: 3000 rows make three, the last one ragged)
    for (m, n, k), mode in [((3000, 700, 300), "exact"), ((3000, 700, 300), "tf32"),
                            ((8192, 64, 40), "exact_simt"), ((5000, 260, 70), "exact")]:
        a, b = operands(m, n, k, "normal", seed=m + k)
        c = g.matmul_host(a, b, mode)
        c64, s = oracle.gemm(a, b)
        check_within_bound(c, c64, s, k, mode, f"host chunks {mode} {m}x{n}x{k}")
    # integers, bitwise, with strided host rows (views into wider arrays)
    m, n, k = 2600, 333, 129
    wa = np.full((m, k + 7), np.nan, np.float32)
    wb = np.full((k, n + 3), np.nan, np.float32)
    wc = np.full((m, n + 5), -3.0, np.float32)
    wa[:, :k] = synth.small_integers((m, k), 91)
    wb[:, :n] = synth.small_integers((k, n), 92)
    for mode in ("exact", "tf32"):
        g.matmul_host(wa[:, :k], wb[:, :n], mode, out=wc[:, :n])
        assert np.array_equal(wc[:, :n].astype(np.float64), oracle.gemm(wa[:, :k], wb[:, :n])[0])
        assert np.all(wc[:, n:] == -3.0), "write outside C's columns"


def test_host_entry_point_long_k(g):
    # the host entry with K past 2048 (row chunks of 1024+ rows, ragged K):
    # within the bound on random data, bitwise on integers with strided host
    # rows
    for (m, n, k), mode in [((2100, 300, 2500), "exact"), ((2100, 300, 2500), "tf32"),
                            ((1100, 260, 2053), "exact_simt")]:
        a, b = operands(m, n, k, "normal", seed=m + n + k)
        c = g.matmul_host(a, b, mode)
        c64, s = oracle.gemm(a, b)
        check_within_bound(c, c64, s, k, mode, f"host long k {mode} {m}x{n}x{k}")
    m, n, k = 1100, 129, 2053
    wa = np.full((m, k + 5), np.nan, np.float32)
    wb = np.full((k, n + 3), np.nan, np.float32)
    wc = np.full((m, n + 2), -7.0, np.float32)
    wa[:, :k] = synth.small_integers((m, k), 93)
    wb[:, :n] = synth.small_integers((k, n), 94)
    expect64 = oracle.gemm(wa[:, :k], wb[:, :n])[0]
    for mode in ("exact", "tf32", "exact_simt"):
        g.matmul_host(wa[:, :k], wb[:, :n], mode, out=wc[:, :n])
        assert np.array_equal(wc[:, :n].astype(np.float64), expect64), mode
        assert np.all(wc[:, n:] == -7.0), "write outside C's columns"


@pytest.mark.parametrize("m,n,k", [(260, 1028, 70), (516, 2048, 300), (258, 1028, 70)])
def test_simt_transposed_staging(g, m, n, k):
    # exact_simt with A stored M x K and N >= 1024 first transposes A into a
    # pooled workspace and stages it K x M (16-byte copies); the result must
    # equal, bit for bit, the kernel run directly on A stored K x M (the same
    # k order per output), and meet the FP32 bound. M not a multiple of 4
    # (258) keeps the direct path.
    a, b = operands(m, n, k, "normal", seed=m + n)
    c, _ = run(g, a, b, "exact_simt")
    c64, s = oracle.gemm(a, b)
    check_within_bound(c, c64, s, k, "exact_simt", f"simt {m}x{n}x{k}")
    da_t = to_dev(np.ascontiguousarray(a.T))
    db = to_dev(b)
    dc = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = g.gemm_f32_general(g.ROW_MAJOR, 1, 0, m, n, k, 1.0, da_t.data_ptr(), m, db.data_ptr(), n,
                            0.0, dc.data_ptr(), n, g.EXACT_SIMT, g.KERNEL_AUTO, stream)
    assert st == g.OK, g.gemm_f32_status_string(st)
    assert np.array_equal(dc.cpu().numpy(), c), "transposed staging changed the result"


def test_host_entry_point_streamed(g):
    # Exact mode from K = 16 runs as one GEMM launch fed while it runs (a
    # ready word per block of up to 1024 rows of A and per half of B's k
    # range, a done counter per block of C); tf32 mode takes the row chunks,
    # checked here on the same shapes. Shapes: fewer rows than one block, a
    # ragged last block, N not a multiple of 256, K just below and just above
    # the 512 from which B goes in two halves, K = 16 in exact mode and K = 4
    # in tf32 mode (random data meets the stated TF32 bound from K = 2 on:
    # one truncated product may be off by 2**-9; K = 1 is checked on integers
    # below); each shape twice (a new epoch each call), and a larger call
    # after smaller ones (the words reallocated).
    cases = [((100, 300, 16), "exact"), ((257, 513, 511), "exact"), ((257, 513, 512), "tf32"),
             ((600, 100, 4), "tf32"), ((1300, 260, 544), "exact"), ((300, 40, 2100), "tf32"),
             ((5200, 520, 700), "exact"), ((5200, 520, 700), "tf32")]
    for (m, n, k), mode in cases:
        a, b = operands(m, n, k, "normal", seed=m + n + k + 1)
        c64, s = oracle.gemm(a, b)
        for rep in range(2):
            c = g.matmul_host(a, b, mode)
            check_within_bound(c, c64, s, k, mode, f"host streamed {mode} {m}x{n}x{k} #{rep}")
    # integers, bitwise, alternating modes back to back; and K = 1 in tf32 mode
    for (m, n, k), modes in [((777, 300, 1000), ("exact", "tf32", "exact", "tf32")),
                             ((600, 100, 1), ("tf32",))]:
        a, b = synth.small_integers((m, k), 95), synth.small_integers((k, n), 96)
        expect64 = oracle.gemm(a, b)[0]
        for mode in modes:
            c = g.matmul_host(a, b, mode).astype(np.float64)
            assert np.array_equal(c, expect64), f"{mode} {m}x{n}x{k}"


def test_host_fed_launch_missing_block_times_out(g):
    # gemm_f32_host's fed launch with the ready word of A's last block never
    # written: the kernel's waits for it run out (20 ms), its CTAs raise every
    # done counter so the copies of C go ahead, and the call returns
    # GEMM_ERR_TIMEOUT; a correct call follows on the same context
    m, n, k = 1300, 520, 544
    a, b = operands(m, n, k, "normal", seed=5)
    # pinned host buffers: the copies are asynchronous, so the host's own
    # bounded wait for them stays in force
    ha = torch.from_numpy(a).pin_memory()
    hb = torch.from_numpy(b).pin_memory()
    hc = torch.full((m, n), float("nan"), dtype=torch.float32).pin_memory()
    st = g.gemm_f32_selftest_host_missing_block(m, n, k, ha.data_ptr(), k, hb.data_ptr(), n,
                                                hc.data_ptr(), n, 20_000_000)
    assert st == g.ERR_TIMEOUT, g.gemm_f32_status_string(st)
    c = g.matmul_host(a, b, "exact")
    c64, s = oracle.gemm(a, b)
    check_within_bound(c, c64, s, k, "exact", "host call after the missing-block self-test")


@pytest.mark.parametrize("mode", ["exact", "tf32"])
def test_host_entry_point_full_size(g, mode):
    # 4096^3 through gemm_f32_host, the bench's end-to-end workload: every
    # 256-row block of C checked on its first and last row and one between,
    # against the oracle's rows
    a, b, _ = config_operands("c4")
    c = g.matmul_host(a, b, mode)
    rows = sorted({r for blk in range(0, 4096, 256) for r in (blk, blk + 131, blk + 255)})
    c64, s = oracle.gemm_rows(a, b, rows)
    check_within_bound(c[rows], c64, s, 4096, mode, f"host 4096^3 {mode}")
    assert np.isfinite(c).all()


def test_probe_peaks_are_plausible(g):
    # MMA-only and FFMA-only probe kernels: rates between half and twice the
    # nominal GB300 figures (1.1 PFLOP/s dense TF32; 152 SMs x 128 lanes x 2
    # flops x 2.07 GHz = 80.5 TFLOP/s FP32), SM clocks at most the maximum
    # (2070 MHz, a little slack for the two clocks' rounding), and the FP32
    # rate within 10 % of what 128 lanes per SM give at the clock it reports
    st, tf32, fp32, tf32_mhz, fp32_mhz = g.gemm_f32_measure_peaks()
    assert st == g.OK, g.gemm_f32_status_string(st)
    assert 550.0 < tf32 < 2200.0, tf32
    assert 40.0 < fp32 < 161.0, fp32
    assert 500.0 < tf32_mhz < 2100.0 and 500.0 < fp32_mhz < 2100.0, (tf32_mhz, fp32_mhz)
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    at_clock = sms * 128 * 2 * fp32_mhz * 1e6 / 1e12
    assert 0.9 * at_clock < fp32 < 1.1 * at_clock, (fp32, at_clock)


def test_bounded_wait_times_out_cleanly(g):
    stream = torch.cuda.current_stream().cuda_stream
    assert g.gemm_f32_selftest_wait_timeout(20_000_000, stream) == g.ERR_TIMEOUT
    # status was cleared by the read, and the context still works
    assert g.gemm_f32_poll_device_status(stream) == g.OK
    a, b = operands(128, 256, 64, "uniform", seed=2)
    c, _ = run(g, a, b, "exact", "tc_tma")
    c64, s = oracle.gemm(a, b)
    check_within_bound(c, c64, s, 64, "exact", "after timeout self-test")


@pytest.mark.parametrize("mode,m,n,k,split", [
    ("exact", 512, 512, 128, False),    # four 256 x 256 tiles, each whole on one pair
    ("tf32", 512, 512, 256, False),
    ("exact", 512, 512, 512, True),     # four pairs of one cluster per tile
    ("tf32", 1024, 1024, 1024, True),
])
def test_pair_kernel_abort_path(g, mode, m, n, k, split):
    # the pair kernel's producers stop after one k-block, so its other roles'
    # waits (limit 20 ms) run out: the kernel must report the timeout, let
    # what it issued finish, free TMEM and return, leaving the context usable
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    st, stats = g.gemm_f32_schedule_check(m, n, k, sms // 2, mode + "_pair")
    assert st == g.OK and (stats["cluster_split"] > 1) == split and stats["splits"] == 0, stats
    a, b = operands(m, n, k, "uniform", seed=11)
    da, db = to_dev(a), to_dev(b)
    dc = torch.zeros((m, n), device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = g.gemm_f32_selftest_stalled_gemm(m, n, k, da.data_ptr(), k, db.data_ptr(), n,
                                          dc.data_ptr(), n, g.MODES[mode], 20_000_000, s)
    assert st == g.ERR_TIMEOUT, g.gemm_f32_status_string(st)
    assert g.gemm_f32_poll_device_status(s) == g.OK
    c, _ = run(g, a, b, mode, "tc_tma")
    c64, sc = oracle.gemm(a, b)
    check_within_bound(c, c64, sc, k, mode, f"{mode} after the stalled pair kernel")


@pytest.mark.parametrize("mode,m,n,k", [("exact", 2048, 1280, 2048), ("tf32", 1280, 2048, 8192)])
def test_stalled_gemm_refuses_workspace_splits(g, mode, m, n, k):
    # 40 unit tiles on 76 pairs: split through the workspace, which the
    # self-test does not take; refused before anything runs
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    st, stats = g.gemm_f32_schedule_check(m, n, k, sms // 2, mode + "_pair")
    assert st == g.OK and stats["splits"] == 1, stats
    la = torch.zeros((m, k), device="cuda")
    lb = torch.zeros((k, n), device="cuda")
    dc = torch.zeros((m, n), device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert g.gemm_f32_selftest_stalled_gemm(m, n, k, la.data_ptr(), k, lb.data_ptr(), n,
                                            dc.data_ptr(), n, g.MODES[mode], 20_000_000,
                                            s) == g.ERR_INVALID_ARG


# ---------------------------------------------------------- full sizes --

# Oracle product of the current workload, computed once and shared by its
# modes, which run one after another (8192 x 11008 x 4096 takes about 25 s on
# 16 host cores and 1.4 GB for C64 and S).
_ORACLE_CACHE = {}


def _oracle_product(cfg, a, b):
    if cfg not in _ORACLE_CACHE:
        _ORACLE_CACHE.clear()
        _ORACLE_CACHE[cfg] = oracle.gemm(a, b)
    return _ORACLE_CACHE[cfg]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("cfg", ["c1", "c2", "c3", "c5a"])
def test_config_full_comparison(g, cfg, mode):
    a, b, c = config_operands(cfg)
    out, _ = run(g, a, b, mode)
    c64, s = _oracle_product(cfg, a, b)
    check_within_bound(out, c64, s, c["K"], mode, f"{cfg} {mode}")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("cfg", ["c4", "c5b"])
def test_config_full_size(g, cfg, mode):
    # full-size workload in the benchmark's launch configuration (dense leading
    # dimensions, default kernel choice, torch's current stream), every element
    # against the fp64 oracle; exact_simt is the FP32 FMA kernel the benchmark
    # also times at 4096^3
    a, b, c = config_operands(cfg)
    out, _ = run(g, a, b, mode)
    assert np.isfinite(out).all()
    c64, s = _oracle_product(cfg, a, b)
    check_within_bound(out, c64, s, c["K"], mode, f"{cfg} {mode}")
