"""gemm_f32_noalloc: the GEMM for callers that may not allocate device memory.

Programs that give almost all device memory to their own allocator, or loops
that must keep the device footprint fixed after set-up, cannot let the GEMM
take its stream-K workspace from the memory pool. gemm_f32_noalloc runs the
same kernels with that workspace in a fixed array inside the library. These
tests call it through the C ABI, twice in a row with different problems (so
the second call starts from the first call's leftovers in the array), and
compare each result with gemm_f32's on the same inputs. This file is
collected last.
"""

import numpy as np
import pytest

import oracle
import synth
from parity import tolerance_factor

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g(gemm_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return gemm_lib


def _both(g, a, b, mode):
    """(C from gemm_f32, C from gemm_f32_noalloc) for the same device inputs."""
    m, k = a.shape
    n = b.shape[1]
    da = torch.from_numpy(a).cuda()
    db = torch.from_numpy(b).cuda()
    ref = torch.full((m, n), float("nan"), device="cuda")
    out = torch.full((m, n), float("nan"), device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert g.gemm_f32(m, n, k, da.data_ptr(), k, db.data_ptr(), n, ref.data_ptr(), n,
                      g.MODES[mode], s) == g.OK
    st = g.gemm_f32_noalloc(m, n, k, da.data_ptr(), k, db.data_ptr(), n, out.data_ptr(), n,
                            g.MODES[mode], s)
    assert st == g.OK, g.gemm_f32_status_string(st)
    assert g.gemm_f32_poll_device_status(s) == g.OK
    return ref.cpu().numpy(), out.cpu().numpy()


def test_noalloc_matches_gemm_f32_on_calls_in_a_row(g):
    # shapes whose output tiles are split between SMs (the workspace is used):
    # 8 tiles each split, then one wave plus split tiles, then the first again
    cases = [((512, 512, 512), "exact"), ((3328, 1536, 512), "tf32"),
             ((512, 512, 512), "exact"), ((1000, 1531, 777), "exact")]
    for (m, n, k), mode in cases:
        a = synth.normal((m, k), m + k)
        b = synth.normal((k, n), n + k)
        ref, out = _both(g, a, b, mode)
        assert np.isfinite(out).all()
        rows = np.unique(np.concatenate([np.arange(0, m, max(1, m // 64)), [m - 1]]))
        _, s = oracle.gemm_rows(a, b, rows)
        tol = tolerance_factor(mode, k) * s
        diff = np.abs(out[rows].astype(np.float64) - ref[rows].astype(np.float64))
        assert np.all(diff <= tol), f"{mode} {m}x{n}x{k}: max diff {diff.max():.3e}"
