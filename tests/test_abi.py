"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and validates arguments and picks kernels on the host
before touching CUDA."""

import ctypes
import os

import pytest

EXPECTED = {
    "gemm_f32", "gemm_f32_ex", "gemm_f32_select", "gemm_f32_host", "gemm_f32_status_string",
    "gemm_f32_poll_device_status", "gemm_f32_selftest_wait_timeout", "gemm_f32_noalloc",
    "gemm_f32_general", "reduce_f32_sum", "gemm_f32_measure_peaks", "gemm_f32_schedule_check",
    "gemm_f32_selftest_stalled_gemm", "gemm_f32_checked_build", "gemm_f32_take_index_fault",
    "gemm_f32_index_site_name", "gemm_f32_selftest_index_check",
    "gemm_f32_selftest_host_missing_block",
}

# Fake, never dereferenced, 256-byte aligned "device" addresses for host-only paths.
PA, PB, PC = 0x10000000, 0x20000000, 0x30000000


def test_header_declares_expected_symbols(gemm_lib):
    assert set(gemm_lib.declared_symbols()) >= EXPECTED


def test_library_exports_every_declared_symbol(gemm_lib):
    lib = ctypes.CDLL(gemm_lib.LIB_PATH)
    for name in gemm_lib.declared_symbols():
        assert hasattr(lib, name), f"{name} declared in include/gemm_f32.h but not exported"


def test_status_strings(gemm_lib):
    names = ["GEMM_OK", "GEMM_ERR_INVALID_ARG", "GEMM_ERR_UNSUPPORTED_DEVICE", "GEMM_ERR_LAUNCH",
             "GEMM_ERR_TIMEOUT", "GEMM_ERR_ALIAS", "GEMM_ERR_INDEX"]
    for code, name in enumerate(names):
        assert gemm_lib.gemm_f32_status_string(code) == name
    assert gemm_lib.gemm_f32_status_string(99) == "GEMM_ERR_UNKNOWN"


@pytest.mark.parametrize("args", [
    dict(M=-1), dict(N=-1), dict(K=-1),
    dict(lda=63), dict(ldb=31), dict(ldc=31),          # leading dimension below the width
    dict(mode=3), dict(mode=-1),
    dict(A=0), dict(B=0), dict(C=0),                   # null with non-zero extents
    dict(A=PA + 2), dict(C=PC + 1),                    # not 4-byte aligned
    dict(M=1 << 31), dict(lda=1 << 31),                # beyond the 2^31 element limit
    dict(M=(1 << 31) - 1, ldc=(1 << 31) - 1),          # spans beyond 2^44 elements
    dict(M=(1 << 31) - 1, lda=(1 << 31) - 1),
    dict(K=(1 << 31) - 1, lda=(1 << 31) - 1, ldb=(1 << 31) - 1),
])
def test_invalid_arguments_rejected_before_any_cuda_call(gemm_lib, args):
    a = dict(M=16, N=32, K=64, A=PA, lda=64, B=PB, ldb=32, C=PC, ldc=32, mode=0)
    a.update(args)
    st = gemm_lib.gemm_f32(a["M"], a["N"], a["K"], a["A"], a["lda"], a["B"], a["ldb"], a["C"],
                           a["ldc"], a["mode"], 0)
    assert st == gemm_lib.ERR_INVALID_ARG


def test_alias_rejected(gemm_lib):
    # C overlapping A, then C overlapping B
    assert gemm_lib.gemm_f32(64, 64, 64, PA, 64, PB, 64, PA + 4 * 100, 64, 0, 0) == gemm_lib.ERR_ALIAS
    assert gemm_lib.gemm_f32(64, 64, 64, PA, 64, PB, 64, PB + 4 * 4032, 64, 0, 0) == gemm_lib.ERR_ALIAS
    # adjacent but not overlapping is fine for validation (selection succeeds)
    assert gemm_lib.gemm_f32_select(64, 64, 64, PA, 64, PA + 4 * 64 * 64, 64, PA + 8 * 64 * 64, 64,
                                    0, 0) > 0


def test_empty_outputs_are_noops(gemm_lib):
    # M == 0 or N == 0: nothing to do, OK without any CUDA call (null pointers allowed)
    assert gemm_lib.gemm_f32(0, 32, 64, 0, 64, 0, 32, 0, 32, 0, 0) == gemm_lib.OK
    assert gemm_lib.gemm_f32(16, 0, 64, 0, 64, 0, 1, 0, 1, 1, 0) == gemm_lib.OK


def test_kernel_selection(gemm_lib):
    sel = gemm_lib.gemm_f32_select
    E, T, S = gemm_lib.EXACT, gemm_lib.TF32, gemm_lib.EXACT_SIMT
    # TMA-legal operands go to the TMA-fed tensor-core kernel in both TC modes
    assert sel(4096, 4096, 4096, PA, 4096, PB, 4096, PC, 4096, E, 0) == gemm_lib.KERNEL_TC_TMA
    assert sel(4096, 4096, 4096, PA, 4096, PB, 4096, PC, 4096, T, 0) == gemm_lib.KERNEL_TC_TMA
    # the ragged workload (row pitches 3108 and 6124 bytes, which TMA cannot
    # read) and a misaligned base still take the TMA-fed kernel: the
    # operands are copied into a workspace with 16-byte pitches first
    assert sel(1000, 1531, 777, PA, 777, PB, 1531, PC, 1531, E, 0) == gemm_lib.KERNEL_TC_TMA
    assert sel(1000, 1531, 777, PA, 777, PB, 1531, PC, 1531, T, 0) == gemm_lib.KERNEL_TC_TMA
    assert sel(64, 64, 64, PA + 4, 64, PB, 64, PC, 64, T, 0) == gemm_lib.KERNEL_TC_TMA
    # exact mode with K < 16 uses the FP32 FMA kernel; EXACT_SIMT always does
    assert sel(64, 64, 15, PA, 16, PB, 64, PC, 64, E, 0) == gemm_lib.KERNEL_SIMT
    assert sel(64, 64, 16, PA, 16, PB, 64, PC, 64, E, 0) == gemm_lib.KERNEL_TC_TMA
    assert sel(4096, 4096, 4096, PA, 4096, PB, 4096, PC, 4096, S, 0) == gemm_lib.KERNEL_SIMT
    # forced kernels: SIMT cannot serve TF32 (accuracy class); TMA takes any
    # strides (through the copy)
    assert sel(64, 64, 64, PA, 64, PB, 64, PC, 64, T, gemm_lib.KERNEL_SIMT) == -gemm_lib.ERR_INVALID_ARG
    assert sel(64, 64, 64, PA, 65, PB, 64, PC, 64, T, gemm_lib.KERNEL_TC_TMA) == gemm_lib.KERNEL_TC_TMA
    assert sel(64, 64, 64, PA, 64, PB, 64, PC, 64, E, gemm_lib.KERNEL_TC_LSU) == gemm_lib.KERNEL_TC_LSU
    assert sel(64, 64, 64, PA, 64, PB, 64, PC, 64, S, gemm_lib.KERNEL_TC_LSU) == -gemm_lib.ERR_INVALID_ARG
    assert sel(64, 64, 64, PA, 64, PB, 64, PC, 64, E, 9) == -gemm_lib.ERR_INVALID_ARG
    # invalid arguments are reported as negative status codes
    assert sel(-1, 64, 64, PA, 64, PB, 64, PC, 64, E, 0) == -gemm_lib.ERR_INVALID_ARG


def _general(gemm_lib, **kw):
    a = dict(order=0, transa=0, transb=0, M=16, N=32, K=64, alpha=1.0, A=PA, lda=64, B=PB, ldb=32,
             beta=0.0, C=PC, ldc=32, mode=0, kernel=0)
    a.update(kw)
    return gemm_lib.gemm_f32_general(a["order"], a["transa"], a["transb"], a["M"], a["N"], a["K"],
                                     a["alpha"], a["A"], a["lda"], a["B"], a["ldb"], a["beta"],
                                     a["C"], a["ldc"], a["mode"], a["kernel"], 0)


@pytest.mark.parametrize("args", [
    dict(order=2), dict(order=-1), dict(transa=2), dict(transb=-1),
    # row-major, A stored K x M: lda >= M; B stored N x K: ldb >= K
    dict(transa=1, lda=15), dict(transb=1, ldb=63), dict(transb=1, ldb=32),
    # column-major: lda >= M (A is M x K), ldb >= K (B is K x N), ldc >= M
    dict(order=1, lda=15), dict(order=1, lda=16, ldb=63), dict(order=1, lda=16, ldb=64, ldc=15),
    dict(order=1, transa=1, lda=63, ldb=64, ldc=16),   # A stored K x M column-major: lda >= K
    dict(mode=3), dict(kernel=9), dict(M=-1),
    dict(transa=1, lda=16, mode=1, kernel=1),          # SIMT cannot serve TF32
])
def test_general_invalid_arguments_rejected(gemm_lib, args):
    assert _general(gemm_lib, **args) == gemm_lib.ERR_INVALID_ARG


def test_general_alias_uses_stored_extents(gemm_lib):
    # B stored N x K (transb) with pitch ldb spans (N - 1) * ldb + K elements:
    # C on its last element overlaps.
    n, k = 32, 64
    last = (n - 1) * k + k - 1
    assert _general(gemm_lib, transb=1, N=n, K=k, ldb=k, C=PB + 4 * last, ldc=n,
                    M=1) == gemm_lib.ERR_ALIAS
    # A stored K x M (transa), pitch lda = M: (K - 1) * M + M elements.
    assert _general(gemm_lib, transa=1, M=16, K=64, A=PA, lda=16, C=PA + 4 * 1023,
                    ldc=32) == gemm_lib.ERR_ALIAS


def test_general_valid_layouts_pass_validation_without_gpu(gemm_lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    fine = (gemm_lib.ERR_LAUNCH, gemm_lib.ERR_UNSUPPORTED_DEVICE)
    assert _general(gemm_lib, transa=1, lda=16) in fine
    assert _general(gemm_lib, transa=1, lda=17, kernel=2) in fine  # A copied for the TMA kernel
    assert _general(gemm_lib, transa=1, lda=16, kernel=2, B=PB + 4) in fine  # and B
    assert _general(gemm_lib, transb=1, ldb=64) in fine
    assert _general(gemm_lib, order=1, lda=16, ldb=64, ldc=16) in fine
    assert _general(gemm_lib, order=1, transa=1, transb=1, lda=64, ldb=32, ldc=16) in fine
    assert _general(gemm_lib, alpha=0.0, beta=2.0) in fine
    # just past the stored N x K extent of B (inside a K x N reading of it)
    assert _general(gemm_lib, transb=1, N=32, K=64, ldb=64, C=PB + 4 * 32 * 64, ldc=32,
                    M=1) in fine
    assert _general(gemm_lib, transa=1, M=16, K=64, A=PA, lda=16, C=PA + 4 * 1024,
                    ldc=32) in fine


@pytest.mark.parametrize("args", [
    dict(n=-1), dict(n=(1 << 40) + 1), dict(groups=-1), dict(groups=65536),
    dict(out=0), dict(out=PC + 2), dict(x=0), dict(x=PA + 1),
])
def test_reduce_invalid_arguments_rejected(gemm_lib, args):
    a = dict(n=1000, x=PA, out=PC, groups=0)
    a.update(args)
    assert gemm_lib.reduce_f32_sum(a["n"], a["x"], a["out"], a["groups"]) == gemm_lib.ERR_INVALID_ARG


def test_reduce_alias_rejected(gemm_lib):
    assert gemm_lib.reduce_f32_sum(1000, PA, PA + 4 * 999, 0) == gemm_lib.ERR_ALIAS
    assert gemm_lib.reduce_f32_sum(1000, PA, PA + 4 * 500, 7) == gemm_lib.ERR_ALIAS


def test_reduce_valid_call_without_gpu_fails_cleanly(gemm_lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    fine = (gemm_lib.ERR_LAUNCH, gemm_lib.ERR_UNSUPPORTED_DEVICE)
    assert gemm_lib.reduce_f32_sum(1000, PA, PA + 4 * 1000, 0) in fine
    assert gemm_lib.reduce_f32_sum(0, 0, PC, 0) in fine


def test_measure_peaks_without_gpu_fails_cleanly(gemm_lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st, _, _, _, _ = gemm_lib.gemm_f32_measure_peaks()
    assert st in (gemm_lib.ERR_LAUNCH, gemm_lib.ERR_UNSUPPORTED_DEVICE)


def test_valid_call_without_gpu_fails_cleanly(gemm_lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = gemm_lib.gemm_f32(64, 64, 64, PA, 64, PB, 64, PC, 64, 0, 0)
    assert st in (gemm_lib.ERR_LAUNCH, gemm_lib.ERR_UNSUPPORTED_DEVICE)


def test_missing_library_fails_loudly(gemm_lib, monkeypatch, tmp_path):
    import dense_fp32_gemm_major_gb300 as g

    monkeypatch.setattr(g, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(g, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        g.gemm_f32(1, 1, 1, PA, 1, PB, 1, PC, 1, 0, 0)


def test_headers_compile_and_link_as_c(gemm_lib, tmp_path):
    # The boundary is a C ABI: the public headers must compile as strict C99
    # and a C program must link against the library and call it (host-only
    # entry points here, so no GPU is needed).
    import shutil
    import subprocess

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not installed")
    src = tmp_path / "abi.c"
    src.write_text(r'''
#include <stdio.h>
#include "gemm_f32.h"
#include "reduce_f32.h"
int main(void) {
  int64_t stats[9];
  int st = gemm_f32_schedule_check(4096, 4096, 4096, 76, GEMM_SCHEDULE_EXACT_PAIR, stats);
  int sel = gemm_f32_select(64, 64, 64, (const float *)0x10000000, 64,
                            (const float *)0x20000000, 64, (float *)0x30000000, 64,
                            GEMM_F32_EXACT, GEMM_KERNEL_AUTO);
  printf("%d %lld %d %s\n", st, (long long)stats[0], sel, gemm_f32_status_string(GEMM_ERR_ALIAS));
  return 0;
}
''')
    lib_dir = os.path.dirname(gemm_lib.LIB_PATH)
    exe = tmp_path / "abi"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", gemm_lib.INCLUDE_DIR, str(src), "-L", lib_dir, "-lgemm_f32",
                    f"-Wl,-rpath,{lib_dir}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    assert out == ["0", "256", str(gemm_lib.KERNEL_TC_TMA), "GEMM_ERR_ALIAS"]


def test_stalled_gemm_self_test_validates_on_the_host(gemm_lib):
    # argument errors come back before any CUDA call: limit out of range,
    # a mode without a pair kernel, bad sizes
    g = gemm_lib
    args = (512, 512, 256, PA, 256, PB, 512, PC, 512)
    assert g.gemm_f32_selftest_stalled_gemm(*args, g.EXACT, 10, 0) == g.ERR_INVALID_ARG
    assert g.gemm_f32_selftest_stalled_gemm(*args, g.EXACT_SIMT, 20_000_000, 0) == g.ERR_INVALID_ARG
    assert g.gemm_f32_selftest_stalled_gemm(512, 512, 256, PA, 255, PB, 512, PC, 512, g.TF32,
                                            20_000_000, 0) == g.ERR_INVALID_ARG


def test_checked_library_exports_every_declared_symbol(gemm_lib, checked_lib):
    for name in gemm_lib.declared_symbols():
        assert hasattr(checked_lib, name), f"{name} not exported by the checked build"
    assert gemm_lib.gemm_f32_checked_build() == 0
    assert gemm_lib.gemm_f32_checked_build(lib=checked_lib) == 1


def test_index_site_names(gemm_lib, checked_lib):
    g = gemm_lib
    expected = {g.SITE_C_STORE: "C store", g.SITE_PARTIAL_WRITE: "partial slot write",
                g.SITE_PARTIAL_READ: "partial slot read", g.SITE_COUNTER: "split-tile counter",
                g.SITE_LOAD_A: "A load", g.SITE_LOAD_B: "B load",
                g.SITE_COPY_SRC: "operand copy source", g.SITE_COPY_DST: "operand copy destination",
                g.SITE_REDUCE_IN: "reduction input", g.SITE_REDUCE_PARTIAL: "reduction partial",
                g.SITE_REDUCE_OUT: "reduction output"}
    for lib in (None, checked_lib):
        for code, name in expected.items():
            assert g.gemm_f32_index_site_name(code, lib=lib) == name
        assert g.gemm_f32_index_site_name(g.SITE_BAND, lib=lib).startswith("cluster-split band")
        assert g.gemm_f32_index_site_name(0, lib=lib) == "none"
        assert g.gemm_f32_index_site_name(99, lib=lib) == "unknown"


def test_index_check_entry_points_validate_on_the_host(gemm_lib, checked_lib):
    g = gemm_lib
    args = (64, 64, 64, PA, 64, PB, 64, PC, 64, g.EXACT)
    # the regular build has no checks: its self-test refuses before any CUDA call
    assert g.gemm_f32_selftest_index_check(*args) == g.ERR_INVALID_ARG
    # the checked build validates as gemm_f32 does, and wants M >= 2, K >= 1
    assert g.gemm_f32_selftest_index_check(1, 64, 64, PA, 64, PB, 64, PC, 64, g.EXACT,
                                           lib=checked_lib) == g.ERR_INVALID_ARG
    assert g.gemm_f32_selftest_index_check(64, 64, 64, PA, 63, PB, 64, PC, 64, g.EXACT,
                                           lib=checked_lib) == g.ERR_INVALID_ARG
    assert g.gemm_f32_selftest_index_check(64, 64, 64, PA, 64, PB, 64, PA, 64, g.EXACT,
                                           lib=checked_lib) == g.ERR_ALIAS
    # null outputs are refused before the device is touched
    for lib in (g.library(), checked_lib):
        assert lib.gemm_f32_take_index_fault(None, None, None, None, None) == g.ERR_INVALID_ARG


def test_checked_build_without_gpu_fails_cleanly(gemm_lib, checked_lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    g = gemm_lib
    st = g.gemm_f32_selftest_index_check(64, 64, 64, PA, 64, PB, 64, PC, 64, g.EXACT,
                                         lib=checked_lib)
    assert st in (g.ERR_LAUNCH, g.ERR_UNSUPPORTED_DEVICE)
    st, count, _, _, _ = g.gemm_f32_take_index_fault(lib=checked_lib)
    assert st in (g.ERR_LAUNCH, g.ERR_UNSUPPORTED_DEVICE) and count == 0


def test_host_missing_block_self_test_validates_on_the_host(gemm_lib):
    g = gemm_lib
    args = (512, 512, 256, PA, 256, PB, 512, PC, 512)
    assert g.gemm_f32_selftest_host_missing_block(*args, 10) == g.ERR_INVALID_ARG      # limit
    assert g.gemm_f32_selftest_host_missing_block(*args, 1 << 40) == g.ERR_INVALID_ARG
    assert g.gemm_f32_selftest_host_missing_block(512, 512, 8, PA, 8, PB, 512, PC, 512,
                                                  20_000_000) == g.ERR_INVALID_ARG      # K < 16
    assert g.gemm_f32_selftest_host_missing_block(512, 512, 256, PA, 255, PB, 512, PC, 512,
                                                  20_000_000) == g.ERR_INVALID_ARG
