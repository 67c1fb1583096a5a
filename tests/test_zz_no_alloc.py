"""gemm_f32_noalloc: the GEMM for callers that may not allocate device memory.

Programs that give almost all device memory to their own allocator at
start-up, or loops that must keep the device footprint fixed once set up,
cannot let the GEMM take its stream-K workspace (partial sums of output tiles
whose k range is shared between SMs) from a memory pool. gemm_f32_noalloc runs
the same kernels with that workspace in a fixed array inside the library.

These tests call it through the C ABI on shapes whose tiles are split (the
array is really used), on both TMA-fed pair kernels and on the plain-load
kernel, several calls back to back on one stream with no synchronisation in
between, so that each call starts from the counters and partial tiles the
previous one left in the array. Every result is compared with the fp64
oracle, element by element, within the mode's bound; the device's free memory
must not change across the calls. This file is collected last.
"""

import numpy as np
import pytest

import oracle
import synth
from parity import check_within_bound

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

# (M, N, K, mode, lda padding, schedule kind). A pitch that is not a multiple
# of 4 floats sends the call to the plain-load kernel (no operand copy may be
# made without allocating). Each shape has more unit tiles than half the CTA
# pairs, so its tiles are split through the workspace (problems with fewer
# tiles split inside a cluster and need none). Workspace of each call on 76
# CTA pairs (152 SMs): 38, 38, 38, 19 and 8 MiB of partial tiles.
SEQUENCE = [
    (2048, 1280, 2048, "exact", 0, "exact_pair"),  # 3xTF32 pairs: 40 tiles, 3 parts each
    (2048, 1280, 2048, "exact", 0, "exact_pair"),  # the same again: counters left counted up
    (1280, 2048, 8192, "tf32", 0, "tf32_pair"),    # one TF32 pass on pairs, 3 parts a tile
    (1000, 1531, 777, "exact", 0, "exact_lsu"),    # lda 777: plain-load 3xTF32 kernel
    (2560, 2048, 1024, "exact", 0, "exact_pair"),  # a full wave whole, the rest split
    (1024, 1024, 1024, "exact", 0, "exact_pair_cs"),  # 16 tiles: split inside clusters,
    (1024, 1024, 1024, "tf32", 0, "tf32_pair_cs"),    # no workspace at all
]
# One call per kernel with a small workspace (6.5, 2 and 1.5 MiB) before the
# memory is measured: a first launch may load code, which is not the GEMM
# allocating, and a pool-backed workspace would then have to grow for the
# larger workspaces of SEQUENCE.
WARMUP = [
    (3328, 1536, 4096, "exact", 0, "exact_pair"),
    (3328, 1536, 4096, "tf32", 0, "tf32_pair"),
    (200, 100, 2000, "exact", 3, "exact_lsu"),
    (512, 512, 512, "exact", 0, "exact_pair_cs"),
    (512, 512, 1024, "tf32", 0, "tf32_pair_cs"),
]


@pytest.fixture(scope="module")
def g(gemm_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return gemm_lib


def _prepare(case, seed):
    """Host operands, device buffers (A with its padded pitch) and a NaN C."""
    m, n, k, mode, pad, _ = case
    a = synth.normal((m, k), seed)
    b = synth.normal((k, n), seed + 1)
    lda = k + pad
    da = torch.full((m, lda), float("nan"), device="cuda")
    da[:, :k] = torch.from_numpy(a).cuda()
    db = torch.from_numpy(b).cuda()
    dc = torch.full((m, n), float("nan"), device="cuda")
    return dict(case=case, a=a, b=b, da=da, lda=lda, db=db, dc=dc)


def _call(g, job, stream):
    m, n, k, mode, _, _ = job["case"]
    st = g.gemm_f32_noalloc(m, n, k, job["da"].data_ptr(), job["lda"], job["db"].data_ptr(), n,
                            job["dc"].data_ptr(), n, g.MODES[mode], stream)
    assert st == g.OK, g.gemm_f32_status_string(st)


def test_noalloc_split_tiles_match_oracle_without_allocating(g):
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    # every shape splits tiles between SMs through the workspace on this
    # device (CTA pairs: the library runs at most sms / 2 of them, fewer if
    # fewer fit at once)
    for m, n, k, mode, pad, kind in WARMUP + SEQUENCE:
        workers = sms if kind.endswith("lsu") else sms // 2
        for w in (workers, workers - 4):
            st, stats = g.gemm_f32_schedule_check(m, n, k, w, kind.replace("_cs", ""))
            if kind.endswith("_cs"):
                ok = stats["splits"] == 0 and stats["cluster_split"] >= 2
            else:
                ok = stats["splits"] == 1 and stats["cluster_split"] == 1
            assert st == g.OK and ok, (m, n, k, kind, w, stats)

    s = torch.cuda.current_stream().cuda_stream
    warm = [_prepare(c, 40 + i) for i, c in enumerate(WARMUP)]
    jobs = [_prepare(c, 60 + 2 * i) for i, c in enumerate(SEQUENCE)]
    jobs[1] = dict(jobs[0], dc=torch.full_like(jobs[0]["dc"], float("nan")))  # same inputs
    for job in warm:
        _call(g, job, s)
    torch.cuda.synchronize()
    assert g.gemm_f32_poll_device_status(s) == g.OK
    free_before, _ = torch.cuda.mem_get_info()

    for job in jobs:  # back to back: no synchronisation between the calls
        _call(g, job, s)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert g.gemm_f32_poll_device_status(s) == g.OK
    assert free_after == free_before, f"device memory changed by {free_before - free_after} bytes"

    for job in warm + jobs:
        m, n, k, mode, _, kind = job["case"]
        c64, sc = oracle.gemm(job["a"], job["b"])
        check_within_bound(job["dc"].cpu().numpy(), c64, sc, k, mode,
                           f"noalloc {kind} {mode} {m}x{n}x{k}")
    # split tiles are summed in a fixed order: the repeated call is bitwise equal
    c0 = jobs[0]["dc"].cpu().numpy()
    c1 = jobs[1]["dc"].cpu().numpy()
    assert np.array_equal(c0.view(np.uint32), c1.view(np.uint32))


def test_noalloc_rejects_what_it_cannot_run_without_allocating(g):
    # validation is that of gemm_f32: nothing is enqueued on an error
    x = torch.zeros((64, 64), device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert g.gemm_f32_noalloc(64, 64, 64, x.data_ptr(), 64, x.data_ptr(), 64, x.data_ptr(), 64,
                              g.EXACT, s) == g.ERR_ALIAS
    assert g.gemm_f32_noalloc(-1, 64, 64, 0, 64, 0, 64, x.data_ptr(), 64, g.EXACT,
                              s) == g.ERR_INVALID_ARG
