"""Python binding checks that need no GPU: views the library cannot address
as (pointer, leading dimension) are refused before any call into it, so a
reversed, expanded, transposed or overlapping view never makes the library
read or write outside the caller's matrix."""

import numpy as np
import pytest
import torch

import dense_fp32_gemm_major_gb300 as g


def test_rows_rule_accepts_addressable_views():
    base = torch.zeros(8, 12)
    for t in (base, base[:, :5], base[2:6, 3:9], base[:, 4:5], base[3:4], torch.zeros(0, 4),
              torch.zeros(4, 0), base.t()[:, :1]):
        g._check_rows(t.shape, t.stride(0), t.stride(1), "t")


@pytest.mark.parametrize("make", [
    lambda: torch.zeros(1, 4).expand(3, 4),                         # row stride 0
    lambda: torch.zeros(4, 3).t(),                                   # column-major
    lambda: torch.zeros(64).as_strided((5, 8), (4, 1)),             # rows overlap
], ids=["expanded", "transposed", "overlapping"])
def test_rows_rule_refuses_unaddressable_views(make):
    t = make()
    with pytest.raises(ValueError):
        g._check_rows(t.shape, t.stride(0), t.stride(1), "t")


def _host(m, n):
    return np.zeros((m, n), np.float32)


@pytest.mark.parametrize("a, b, out, exc", [
    (_host(6, 4)[::-1], _host(4, 5), None, ValueError),               # reversed rows
    (_host(6, 4), np.zeros((5, 4), np.float32).T, None, ValueError),  # column-major B
    (_host(6, 4), _host(4, 5), _host(5, 6), ValueError),              # out of the wrong shape
    (_host(6, 4), _host(4, 5), _host(6, 5)[:, ::-1], ValueError),     # out with reversed columns
    (_host(6, 4), _host(4, 5), np.zeros((6, 5), np.float64), TypeError),
    (_host(6, 4).astype(np.float64), _host(4, 5), None, TypeError),
    (_host(6, 4), _host(3, 5), None, ValueError),                      # inner dimensions differ
], ids=["reversed-a", "colmajor-b", "out-shape", "out-reversed", "out-dtype", "a-dtype", "inner"])
def test_matmul_host_refuses_before_calling_the_library(a, b, out, exc):
    with pytest.raises(exc):
        g.matmul_host(a, b, "exact", out=out)


def test_matmul_host_refuses_read_only_out():
    out = _host(6, 5)
    out.flags.writeable = False
    with pytest.raises(ValueError):
        g.matmul_host(_host(6, 4), _host(4, 5), "exact", out=out)


def test_matmul_host_refuses_byte_strided_views():
    # a column stride of 6 bytes: not a whole number of elements
    buf = np.zeros(6 * 17, np.float32)
    a = np.lib.stride_tricks.as_strided(buf, shape=(6, 4), strides=(17 * 4, 6))
    with pytest.raises(ValueError):
        g.matmul_host(a, _host(4, 5), "exact")


def test_torch_wrappers_refuse_cpu_tensors():
    with pytest.raises(TypeError):
        g.matmul(torch.zeros(4, 4), torch.zeros(4, 4))
    with pytest.raises(TypeError):
        g.gemm(torch.zeros(4, 4), torch.zeros(4, 4))
    with pytest.raises(TypeError):
        g.vector_sum(torch.zeros(8))
