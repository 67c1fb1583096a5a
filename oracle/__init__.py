"""fp64 oracle for C = A x B (row-major fp32 operands) and for the sum of a
fp32 vector.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package. The CUDA library never
calls it, and it never calls the CUDA library: the two share nothing but the
seeded inputs from ``synth``.

The arithmetic lives in ``gemm_oracle.c`` and ``reduce_oracle.c`` (plain C,
fp64, no blocking); this file compiles them on first use and wraps them with
ctypes. Every function returns
``(C64, S)`` where ``C64[i, j] = sum_k A[i, k] * B[k, j]`` in fp64 and
``S[i, j] = sum_k |A[i, k]| * |B[k, j]|``: the product that
"Optimizing a WebGPU Matmul Kernel using Subgroups", section 1 "Naive", and the
CPU triple loop of "WebGPU 行列積の限界を測る" define.

Pins: tests/test_oracle.py checks this code against hand-worked products
(tests/golden/), identity, permutation and diagonal factors, the all-ones
closed form, linearity, the transpose identity, exact rational brute force and
the integer-valued self-test pattern of "GPU compute shaders" (section "Code").
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "gemm_oracle.c"), os.path.join(_HERE, "reduce_oracle.c")]
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle's C sources into oracle/_build/liboracle.so (OpenMP if
    available)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and all(os.path.getmtime(_LIB) >= os.path.getmtime(f) for f in _SRCS)):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]
    tmp = _LIB + f".tmp{os.getpid()}"
    try:
        subprocess.run(base + ["-fopenmp", "-o", tmp] + _SRCS + ["-lm"], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-o", tmp] + _SRCS + ["-lm"], check=True, capture_output=True,
                       text=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, p = ctypes.c_int64, ctypes.c_void_p
            lib.oracle_gemm_f64.argtypes = [i64, i64, i64, p, i64, p, i64, p, i64, p, i64]
            lib.oracle_gemm_f64.restype = None
            lib.oracle_gemm_rows_f64.argtypes = [i64, p, i64, i64, p, i64, p, i64, p, p]
            lib.oracle_gemm_rows_f64.restype = None
            lib.oracle_gemm_entries_f64.argtypes = [i64, p, p, i64, p, i64, p, i64, p, p]
            lib.oracle_gemm_entries_f64.restype = None
            d = ctypes.c_double
            lib.oracle_gemm_general_rows_f64.argtypes = [ctypes.c_int, ctypes.c_int, i64, p, i64, i64,
                                                         d, p, i64, p, i64, d, p, i64, p, p]
            lib.oracle_gemm_general_rows_f64.restype = None
            lib.oracle_sum_f64.argtypes = [i64, p, p, p]
            lib.oracle_sum_f64.restype = None
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _as_f32_2d(x: np.ndarray, name: str) -> np.ndarray:
    if x.dtype != np.float32 or x.ndim != 2:
        raise TypeError(f"{name} must be a 2-D float32 array")
    if x.strides[1] != 4:
        x = np.ascontiguousarray(x)
    return x


def _ptr(x: np.ndarray) -> int:
    return x.ctypes.data


def _ld(x: np.ndarray) -> int:
    return x.strides[0] // 4 if x.shape[0] > 1 else max(x.shape[1], 1)


def gemm(a: np.ndarray, b: np.ndarray):
    """Full product of a (M x K) and b (K x N): returns (C64, S), both M x N fp64.

    ``a`` and ``b`` may be row-major views with a leading dimension larger than
    their width (their row stride is passed through as lda / ldb).
    """
    a = _as_f32_2d(a, "a")
    b = _as_f32_2d(b, "b")
    m, k = a.shape
    k2, n = b.shape
    if k != k2:
        raise ValueError("inner dimensions differ")
    c64 = np.zeros((m, n), dtype=np.float64)
    s = np.zeros((m, n), dtype=np.float64)
    if m and n:
        _load().oracle_gemm_f64(m, n, k, _ptr(a), _ld(a), _ptr(b), _ld(b),
                                _ptr(c64), max(n, 1), _ptr(s), max(n, 1))
    return c64, s


def gemm_rows(a: np.ndarray, b: np.ndarray, rows):
    """Rows ``rows`` of the product: returns (C64, S), each len(rows) x N."""
    a = _as_f32_2d(a, "a")
    b = _as_f32_2d(b, "b")
    m, k = a.shape
    k2, n = b.shape
    if k != k2:
        raise ValueError("inner dimensions differ")
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    if rows.size and (rows.min() < 0 or rows.max() >= m):
        raise IndexError("row out of range")
    c64 = np.zeros((rows.size, n), dtype=np.float64)
    s = np.zeros((rows.size, n), dtype=np.float64)
    if rows.size and n:
        _load().oracle_gemm_rows_f64(rows.size, _ptr(rows), n, k, _ptr(a), _ld(a),
                                     _ptr(b), _ld(b), _ptr(c64), _ptr(s))
    return c64, s


def gemm_entries(a: np.ndarray, b: np.ndarray, ii, jj):
    """Entries (ii[t], jj[t]) of the product: returns (c64, s) 1-D fp64 arrays."""
    a = _as_f32_2d(a, "a")
    b = _as_f32_2d(b, "b")
    m, k = a.shape
    k2, n = b.shape
    if k != k2:
        raise ValueError("inner dimensions differ")
    ii = np.ascontiguousarray(np.asarray(ii, dtype=np.int64))
    jj = np.ascontiguousarray(np.asarray(jj, dtype=np.int64))
    if ii.shape != jj.shape:
        raise ValueError("ii and jj differ in shape")
    if ii.size and (ii.min() < 0 or ii.max() >= m or jj.min() < 0 or jj.max() >= n):
        raise IndexError("entry out of range")
    c64 = np.zeros(ii.size, dtype=np.float64)
    s = np.zeros(ii.size, dtype=np.float64)
    if ii.size:
        _load().oracle_gemm_entries_f64(ii.size, _ptr(ii), _ptr(jj), k, _ptr(a), _ld(a),
                                        _ptr(b), _ld(b), _ptr(c64), _ptr(s))
    return c64, s


def gemm_general(a: np.ndarray, b: np.ndarray, opb: int = 0, alpha: float = 1.0,
                 beta: float = 0.0, c: np.ndarray | None = None, rows=None, opa: int = 0):
    """Cout = alpha * op(a) @ op(b) + beta * c in fp64, and S = |op(a)| @ |op(b)|.

    op(a) = a (M x K) when opa == 0, or a.T when opa == 1 (a then stored K x M);
    op(b) = b (K x N) when opb == 0, or b.T when opb == 1 (b then stored N x K).
    ``c`` (M x N fp32) is read only when beta != 0. ``rows`` selects output rows
    (default: all). Returns (Cout, S), each len(rows) x N.
    """
    a = _as_f32_2d(a, "a")
    b = _as_f32_2d(b, "b")
    m, k = (a.shape[1], a.shape[0]) if opa else a.shape
    n, kb = (b.shape[1], b.shape[0]) if opb == 0 else (b.shape[0], b.shape[1])
    if k != kb:
        raise ValueError("inner dimensions differ")
    rows = np.arange(m, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    rows = np.ascontiguousarray(rows)
    if beta != 0.0:
        if c is None or c.shape != (m, n):
            raise ValueError("beta != 0 needs c of shape (M, N)")
        c = _as_f32_2d(c, "c")
        cptr, ldc = _ptr(c), _ld(c)
    else:
        cptr, ldc = None, max(n, 1)
    out = np.zeros((rows.size, n), dtype=np.float64)
    s = np.zeros((rows.size, n), dtype=np.float64)
    if rows.size and n:
        _load().oracle_gemm_general_rows_f64(int(opa), int(opb), rows.size, _ptr(rows), n, k,
                                             float(alpha),
                                             _ptr(a), _ld(a), _ptr(b), _ld(b), float(beta), cptr,
                                             ldc, _ptr(out), _ptr(s))
    return out, s


def vector_sum(x: np.ndarray):
    """Sum of a 1-D float32 array in fp64, in index order: returns (s64, S)
    with S = sum |x|. The quantity the per-group tree reduction of "GPU
    compute shaders" computes."""
    if not isinstance(x, np.ndarray) or x.dtype != np.float32 or x.ndim != 1:
        raise TypeError("x must be a 1-D float32 array")
    x = np.ascontiguousarray(x)
    s64 = ctypes.c_double(0.0)
    scale = ctypes.c_double(0.0)
    _load().oracle_sum_f64(x.size, _ptr(x), ctypes.addressof(s64), ctypes.addressof(scale))
    return s64.value, scale.value


def num_threads() -> int:
    """Host threads the oracle's parallel loops use."""
    return int(_load().oracle_num_threads())
