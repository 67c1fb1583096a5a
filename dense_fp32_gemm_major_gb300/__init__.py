"""Python binding of libgemm_f32.so: dense row-major fp32 GEMM on GB300.

Argument marshalling only. Every step of the product runs in the library's
CUDA kernels; there is no CPU or PyTorch fallback. Importing the package does
not need a GPU, but it does need the built library: if libgemm_f32.so is
missing the import fails loudly (build it with ``__graft_entry__.build()`` or
``python -m dense_fp32_gemm_major_gb300._build``).

The entry points mirror include/gemm_f32.h one to one (same names, same
argument order; pointers are plain integers, streams are ``cudaStream_t``
values as integers, 0 = the legacy default stream). ``matmul`` and ``gemm``
are convenience wrappers over ``gemm_f32_ex`` and ``gemm_f32_general`` for
torch CUDA tensors.

``checked_library()`` loads libgemm_f32_checked.so, the same library built
with device-side index checks (see include/gemm_f32.h, "The checked build");
its handle has the same functions, and the wrappers below take it as ``lib``.
"""

from __future__ import annotations

import ctypes
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgemm_f32.so")
LIB_CHECKED_PATH = os.path.join(_PKG, "libgemm_f32_checked.so")
INCLUDE_DIR = os.path.join(os.path.dirname(_PKG), "include")
HEADER_PATH = os.path.join(INCLUDE_DIR, "gemm_f32.h")
HEADERS = [HEADER_PATH, os.path.join(INCLUDE_DIR, "reduce_f32.h")]

# gemm_f32_mode
EXACT, TF32, EXACT_SIMT = 0, 1, 2
MODES = {"exact": EXACT, "tf32": TF32, "exact_simt": EXACT_SIMT}
# gemm_f32_status
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_DEVICE, ERR_LAUNCH, ERR_TIMEOUT, ERR_ALIAS, ERR_INDEX = range(7)
# index-check sites (gemm_f32_take_index_fault)
SITE_C_STORE, SITE_PARTIAL_WRITE, SITE_PARTIAL_READ, SITE_COUNTER, SITE_BAND = range(1, 6)
SITE_LOAD_A, SITE_LOAD_B, SITE_COPY_SRC, SITE_COPY_DST = range(6, 10)
SITE_REDUCE_IN, SITE_REDUCE_PARTIAL, SITE_REDUCE_OUT = range(10, 13)
# fixed scratch of gemm_f32_noalloc
NOALLOC_SCRATCH_BYTES = 40 * 1024 * 1024
# gemm_f32_kernel
KERNEL_AUTO, KERNEL_SIMT, KERNEL_TC_TMA, KERNEL_TC_LSU = range(4)
KERNELS = {"auto": KERNEL_AUTO, "simt": KERNEL_SIMT, "tc_tma": KERNEL_TC_TMA, "tc_lsu": KERNEL_TC_LSU}
# gemm_f32_order, gemm_f32_op
ROW_MAJOR, COL_MAJOR = 0, 1
OP_N, OP_T = 0, 1


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str = "gemm_f32"):
        self.status = status
        super().__init__(f"{what} failed: {gemm_f32_status_string(status)} ({status})")


_lib = None
_lib_checked = None


def _open(path):
    if not os.path.exists(path):
        raise RuntimeError(
            f"{os.path.basename(path)} is not built ({path}); run __graft_entry__.build(). "
            "There is no fallback implementation.")
    lib = ctypes.CDLL(path)
    i64, i32, p = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    sig = [i64, i64, i64, p, i64, p, i64, p, i64]
    lib.gemm_f32.argtypes = sig + [i32, p]
    lib.gemm_f32.restype = i32
    lib.gemm_f32_ex.argtypes = sig + [i32, i32, p]
    lib.gemm_f32_ex.restype = i32
    lib.gemm_f32_select.argtypes = sig + [i32, i32]
    lib.gemm_f32_select.restype = i32
    lib.gemm_f32_host.argtypes = sig + [i32]
    lib.gemm_f32_host.restype = i32
    lib.gemm_f32_noalloc.argtypes = sig + [i32, p]
    lib.gemm_f32_noalloc.restype = i32
    f32 = ctypes.c_float
    lib.gemm_f32_general.argtypes = [i32, i32, i32, i64, i64, i64, f32, p, i64, p, i64, f32, p,
                                     i64, i32, i32, p]
    lib.gemm_f32_general.restype = i32
    lib.reduce_f32_sum.argtypes = [i64, p, p, i32, p]
    lib.reduce_f32_sum.restype = i32
    lib.gemm_f32_status_string.argtypes = [i32]
    lib.gemm_f32_status_string.restype = ctypes.c_char_p
    lib.gemm_f32_measure_peaks.argtypes = [ctypes.POINTER(ctypes.c_double)] * 4
    lib.gemm_f32_measure_peaks.restype = i32
    lib.gemm_f32_poll_device_status.argtypes = [p]
    lib.gemm_f32_poll_device_status.restype = i32
    lib.gemm_f32_selftest_wait_timeout.argtypes = [i64, p]
    lib.gemm_f32_selftest_wait_timeout.restype = i32
    lib.gemm_f32_selftest_stalled_gemm.argtypes = sig + [i32, i64, p]
    lib.gemm_f32_selftest_stalled_gemm.restype = i32
    lib.gemm_f32_selftest_host_missing_block.argtypes = sig + [i64]
    lib.gemm_f32_selftest_host_missing_block.restype = i32
    lib.gemm_f32_schedule_check.argtypes = [i64, i64, i64, i64, i32, ctypes.POINTER(ctypes.c_int64)]
    lib.gemm_f32_schedule_check.restype = i32
    lib.gemm_f32_checked_build.argtypes = []
    lib.gemm_f32_checked_build.restype = i32
    ll = ctypes.POINTER(ctypes.c_longlong)
    lib.gemm_f32_take_index_fault.argtypes = [p, ll, ctypes.POINTER(i32), ll, ll]
    lib.gemm_f32_take_index_fault.restype = i32
    lib.gemm_f32_index_site_name.argtypes = [i32]
    lib.gemm_f32_index_site_name.restype = ctypes.c_char_p
    lib.gemm_f32_selftest_index_check.argtypes = sig + [i32, i32, p]
    lib.gemm_f32_selftest_index_check.restype = i32
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _open(LIB_PATH)
    return _lib


def reload():
    """Drop the cached handles (after a rebuild) and load the library again."""
    global _lib, _lib_checked
    _lib = None
    _lib_checked = None
    return _load()


def library():
    return _load()


def checked_library():
    """The index-checked build (libgemm_f32_checked.so): same functions as
    library(); slower, for debugging and the index-check tests."""
    global _lib_checked
    if _lib_checked is None:
        _lib_checked = _open(LIB_CHECKED_PATH)
    return _lib_checked


def declared_symbols() -> list[str]:
    """Function names declared in the public headers (include/*.h)."""
    names = set()
    for path in HEADERS:
        with open(path) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*((?:gemm|reduce)_f32\w*)\s*\(",
                                text, flags=re.M))
    return sorted(names)


# ------------------------------------------------------------ raw C ABI --

def gemm_f32(M, N, K, A, lda, B, ldb, C, ldc, mode, stream=0) -> int:
    return _load().gemm_f32(M, N, K, A, lda, B, ldb, C, ldc, mode, stream or None)


def gemm_f32_ex(M, N, K, A, lda, B, ldb, C, ldc, mode, kernel, stream=0) -> int:
    return _load().gemm_f32_ex(M, N, K, A, lda, B, ldb, C, ldc, mode, kernel, stream or None)


def gemm_f32_general(order, transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, mode,
                     kernel=KERNEL_AUTO, stream=0) -> int:
    """C = alpha * op(A) op(B) + beta * C (see include/gemm_f32.h)."""
    return _load().gemm_f32_general(order, transa, transb, M, N, K, alpha, A, lda, B, ldb, beta,
                                    C, ldc, mode, kernel, stream or None)


def gemm_f32_select(M, N, K, A, lda, B, ldb, C, ldc, mode, kernel=KERNEL_AUTO) -> int:
    return _load().gemm_f32_select(M, N, K, A, lda, B, ldb, C, ldc, mode, kernel)


def gemm_f32_host(M, N, K, A, lda, B, ldb, C, ldc, mode) -> int:
    return _load().gemm_f32_host(M, N, K, A, lda, B, ldb, C, ldc, mode)


def gemm_f32_noalloc(M, N, K, A, lda, B, ldb, C, ldc, mode, stream=0) -> int:
    """gemm_f32 that allocates no device memory (workspace in a fixed
    NOALLOC_SCRATCH_BYTES array; see include/gemm_f32.h)."""
    return _load().gemm_f32_noalloc(M, N, K, A, lda, B, ldb, C, ldc, mode, stream or None)


def reduce_f32_sum(n, x, out, groups=0, stream=0) -> int:
    """*out = sum of x[0, n) (device pointers; see include/reduce_f32.h)."""
    return _load().reduce_f32_sum(n, x, out, groups, stream or None)


def gemm_f32_status_string(status: int) -> str:
    return _load().gemm_f32_status_string(status).decode()


def gemm_f32_measure_peaks():
    """(status, tf32_tflops, fp32_tflops, tf32_sm_mhz, fp32_sm_mhz) from the
    MMA-only and FFMA-only probe kernels on the current device: each rate and
    the median SM clock its kernel ran at."""
    t, f = ctypes.c_double(0.0), ctypes.c_double(0.0)
    tc, fc = ctypes.c_double(0.0), ctypes.c_double(0.0)
    st = _load().gemm_f32_measure_peaks(ctypes.byref(t), ctypes.byref(f), ctypes.byref(tc),
                                        ctypes.byref(fc))
    return st, t.value, f.value, tc.value, fc.value


def gemm_f32_poll_device_status(stream=0) -> int:
    return _load().gemm_f32_poll_device_status(stream or None)


def gemm_f32_selftest_wait_timeout(timeout_ns: int, stream=0) -> int:
    return _load().gemm_f32_selftest_wait_timeout(timeout_ns, stream or None)


def gemm_f32_selftest_stalled_gemm(M, N, K, A, lda, B, ldb, C, ldc, mode, timeout_ns,
                                   stream=0) -> int:
    return _load().gemm_f32_selftest_stalled_gemm(M, N, K, A, lda, B, ldb, C, ldc, mode,
                                                  timeout_ns, stream or None)


def gemm_f32_checked_build(lib=None) -> int:
    return (lib or _load()).gemm_f32_checked_build()


def gemm_f32_take_index_fault(stream=0, lib=None):
    """(status, count, site, offset, extent): the index-check record since the
    last call, reset (checked build; count is always 0 in the regular one)."""
    count, off, ext = ctypes.c_longlong(0), ctypes.c_longlong(0), ctypes.c_longlong(0)
    site = ctypes.c_int(0)
    st = (lib or _load()).gemm_f32_take_index_fault(stream or None, ctypes.byref(count),
                                                   ctypes.byref(site), ctypes.byref(off),
                                                   ctypes.byref(ext))
    return st, count.value, site.value, off.value, ext.value


def gemm_f32_index_site_name(site: int, lib=None) -> str:
    return (lib or _load()).gemm_f32_index_site_name(site).decode()


def gemm_f32_selftest_index_check(M, N, K, A, lda, B, ldb, C, ldc, mode, kernel=KERNEL_AUTO,
                                  stream=0, lib=None) -> int:
    return (lib or _load()).gemm_f32_selftest_index_check(M, N, K, A, lda, B, ldb, C, ldc, mode,
                                                         kernel, stream or None)


def gemm_f32_selftest_host_missing_block(M, N, K, A, lda, B, ldb, C, ldc, timeout_ns) -> int:
    return _load().gemm_f32_selftest_host_missing_block(M, N, K, A, lda, B, ldb, C, ldc,
                                                        timeout_ns)


SCHEDULE_KINDS = {"exact_pair": 0, "tf32_pair": 1, "exact_lsu": 2, "tf32_lsu": 3}
SCHEDULE_STATS = ("tiles", "k_blocks", "whole_tiles", "sk_share", "sk_clusters", "splits",
                  "max_parts", "clusters", "cluster_split")


def gemm_f32_schedule_check(m: int, n: int, k: int, workers: int, kind):
    """Host-only check of the tile schedule (no GPU): (status, stats dict)."""
    stats = (ctypes.c_int64 * len(SCHEDULE_STATS))()
    kind = SCHEDULE_KINDS[kind] if isinstance(kind, str) else int(kind)
    st = _load().gemm_f32_schedule_check(m, n, k, workers, kind, stats)
    return st, dict(zip(SCHEDULE_STATS, list(stats)))


# ---------------------------------------------------------- conveniences --

def _mode(mode) -> int:
    return MODES[mode] if isinstance(mode, str) else int(mode)


def _kernel(kernel) -> int:
    return KERNELS[kernel] if isinstance(kernel, str) else int(kernel)


def _check_rows(shape, row_stride, col_stride, name):
    """A matrix the library can address as (pointer, leading dimension): unit
    column stride and rows that do not overlap (strides in elements). Views
    that break either rule (expanded, transposed or reversed ones) would make
    the library read or write outside the matrix, so they are refused."""
    rows, cols = int(shape[0]), int(shape[1])
    if rows == 0 or cols == 0:
        return
    if cols > 1 and col_stride != 1:
        raise ValueError(f"{name} must be row-major (unit column stride)")
    if rows > 1 and row_stride < cols:
        raise ValueError(f"{name} has overlapping or reversed rows (row stride {row_stride} "
                         f"for {cols} columns)")


def _check_operand(t, name, device=None):
    import torch

    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or not t.is_cuda or t.dim() != 2:
        raise TypeError(f"{name} must be a 2-D float32 CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, the other operands on {device}")
    _check_rows(t.shape, t.stride(0), t.stride(1), name)


def _ld(t) -> int:
    return max(int(t.stride(0)), int(t.shape[1]), 1) if t.shape[0] > 1 else max(int(t.shape[1]), 1)


def matmul(a, b, mode="exact", out=None, kernel="auto", stream=None):
    """C = A x B for row-major float32 CUDA tensors (stream ordered).

    ``a`` is M x K, ``b`` K x N; ``out`` (M x N, row-major, may have a padded
    row stride) is overwritten and returned. ``stream`` defaults to torch's
    current stream.
    """
    import torch

    _check_operand(a, "a")
    _check_operand(b, "b", a.device)
    m, k = a.shape
    k2, n = b.shape
    if k != k2:
        raise ValueError(f"inner dimensions differ: {tuple(a.shape)} x {tuple(b.shape)}")
    if out is None:
        out = torch.empty((m, n), dtype=torch.float32, device=a.device)
    else:
        _check_operand(out, "out", a.device)
        if tuple(out.shape) != (m, n):
            raise ValueError("out has the wrong shape")
    if stream is None:
        stream = torch.cuda.current_stream(a.device).cuda_stream
    with torch.cuda.device(a.device):
        st = gemm_f32_ex(m, n, k, a.data_ptr(), _ld(a), b.data_ptr(), _ld(b), out.data_ptr(),
                         _ld(out), _mode(mode), _kernel(kernel), stream)
    if st != OK:
        raise GemmError(st)
    return out


def gemm(a, b, out=None, alpha=1.0, beta=0.0, transa=False, transb=False, mode="exact",
         kernel="auto", stream=None):
    """out = alpha * op(a) op(b) + beta * out for row-major float32 CUDA tensors.

    ``a`` is stored M x K, or K x M with ``transa``; ``b`` K x N, or N x K
    with ``transb``. ``out`` (M x N) is read only when beta != 0 and is
    required then. Stream ordered on ``stream`` (default: torch's current
    stream); returns ``out``.
    """
    import torch

    _check_operand(a, "a")
    _check_operand(b, "b", a.device)
    m, k = (a.shape[1], a.shape[0]) if transa else tuple(a.shape)
    k2, n = (b.shape[1], b.shape[0]) if transb else tuple(b.shape)
    if k != k2:
        raise ValueError(f"inner dimensions differ: op(a) is {m} x {k}, op(b) is {k2} x {n}")
    if out is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs out")
        out = torch.empty((m, n), dtype=torch.float32, device=a.device)
    else:
        _check_operand(out, "out", a.device)
        if tuple(out.shape) != (m, n):
            raise ValueError("out has the wrong shape")
    if stream is None:
        stream = torch.cuda.current_stream(a.device).cuda_stream
    with torch.cuda.device(a.device):
        st = gemm_f32_general(ROW_MAJOR, OP_T if transa else OP_N, OP_T if transb else OP_N, m, n,
                              k, float(alpha), a.data_ptr(), _ld(a), b.data_ptr(), _ld(b),
                              float(beta), out.data_ptr(), _ld(out), _mode(mode), _kernel(kernel),
                              stream)
    if st != OK:
        raise GemmError(st, "gemm_f32_general")
    return out


def vector_sum(x, groups=0, out=None, stream=None):
    """Sum of a 1-D float32 CUDA tensor through reduce_f32_sum; returns a
    one-element float32 CUDA tensor (stream ordered)."""
    import torch

    if (not isinstance(x, torch.Tensor) or x.dtype != torch.float32 or not x.is_cuda
            or x.dim() != 1 or (x.numel() > 1 and x.stride(0) != 1)):
        raise TypeError("x must be a contiguous 1-D float32 CUDA tensor")
    if out is None:
        out = torch.empty(1, dtype=torch.float32, device=x.device)
    elif (not isinstance(out, torch.Tensor) or out.dtype != torch.float32
          or out.device != x.device or out.numel() < 1):
        raise TypeError("out must be a float32 tensor of at least one element on x's device")
    if stream is None:
        stream = torch.cuda.current_stream(x.device).cuda_stream
    with torch.cuda.device(x.device):
        st = reduce_f32_sum(x.numel(), x.data_ptr(), out.data_ptr(), int(groups), stream)
    if st != OK:
        raise GemmError(st, "reduce_f32_sum")
    return out


def _check_host(x, name):
    import numpy as np

    if not isinstance(x, np.ndarray) or x.dtype != np.float32 or x.ndim != 2:
        raise TypeError(f"{name} must be a 2-D float32 numpy array")
    if x.strides[0] % 4 or x.strides[1] % 4:
        raise ValueError(f"{name}'s strides are not whole elements")
    _check_rows(x.shape, x.strides[0] // 4, x.strides[1] // 4, name)


def matmul_host(a, b, mode="exact", out=None):
    """C = A x B for host numpy float32 arrays through gemm_f32_host (blocking)."""
    import numpy as np

    _check_host(a, "a")
    _check_host(b, "b")
    m, k = a.shape
    k2, n = b.shape
    if k != k2:
        raise ValueError("inner dimensions differ")
    if out is None:
        out = np.empty((m, n), dtype=np.float32)
    else:
        _check_host(out, "out")
        if out.shape != (m, n):
            raise ValueError("out has the wrong shape")
        if not out.flags.writeable:
            raise ValueError("out is read-only")
    ld = lambda x: max(x.strides[0] // 4, x.shape[1], 1) if x.shape[0] > 1 else max(x.shape[1], 1)
    st = gemm_f32_host(m, n, k, a.ctypes.data, ld(a), b.ctypes.data, ld(b), out.ctypes.data,
                       ld(out), _mode(mode))
    if st != OK:
        raise GemmError(st, "gemm_f32_host")
    return out
