"""Parity of reduce_f32_sum (per-group partial sums and a second dispatch,
as in "GPU compute shaders") against the fp64 oracle, through the C ABI.

Random inputs are checked within the bound the header states; integer-valued
inputs (whose fp32 partial sums are all exact) must match the exact sum
bitwise, and reruns with the same group count must be bit-identical.
"""

import math

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g(gemm_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return gemm_lib


def device_sum(g, x_dev, n, groups=0, offset=0):
    out = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = g.reduce_f32_sum(n, x_dev.data_ptr() + 4 * offset, out.data_ptr(), groups, s)
    assert st == g.OK, g.gemm_f32_status_string(st)
    return float(out.item())


def bound(n, groups, scale):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    G = groups or 4 * sms
    h = math.ceil(n / (1024 * G)) + math.ceil(G / 256) + 24
    return 1.01 * h * 2.0 ** -24 * scale


def test_pages_integer_self_test(g):
    # "GPU compute shaders", section "Code": (37 i mod 101) - 50, n = 10000,
    # 7 groups: the partial sums add up to the plain sum exactly, and a rerun
    # is bit-identical
    n = 10_000
    v = np.array([(i * 37 % 101) - 50 for i in range(n)], dtype=np.float32)
    xd = torch.from_numpy(v).cuda()
    s1 = device_sum(g, xd, n, groups=7)
    assert s1 == oracle.vector_sum(v)[0] == sum((i * 37 % 101) - 50 for i in range(n))
    assert device_sum(g, xd, n, groups=7) == s1
    for groups in (0, 1, 3, 608, 65535):
        assert device_sum(g, xd, n, groups=groups) == s1


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 255, 1023, 1024, 4097, 100_003, (1 << 20) + 3])
@pytest.mark.parametrize("groups", [0, 1, 7, 608, 65535])
@pytest.mark.parametrize("offset", [0, 1, 2])
def test_random_within_bound(g, n, groups, offset):
    x = synth.uniform_pm1((n + offset,), 900 + n % 1000).reshape(-1)
    xd = torch.from_numpy(x).cuda()
    got = device_sum(g, xd, n, groups, offset)
    s64, scale = oracle.vector_sum(x[offset:])
    assert math.isfinite(got)
    assert abs(got - s64) <= bound(n, groups, scale), (got, s64, bound(n, groups, scale))


def test_integers_bitwise_any_grouping(g):
    n = 3_000_001
    x = synth.small_integers((n,), 77).reshape(-1)
    xd = torch.from_numpy(x).cuda()
    s64, _ = oracle.vector_sum(x)
    for groups, offset in ((0, 0), (1, 0), (13, 1), (65535, 3)):
        m = n - offset
        assert device_sum(g, xd, m, groups, offset) == oracle.vector_sum(x[offset:])[0]


def test_closed_forms(g):
    for n in (1, 17, 1 << 20, (1 << 24) - 5):
        assert device_sum(g, torch.ones(n, device="cuda"), n) == float(n)
    # alternating +-1: every group's partial is small and exact
    n = (1 << 21) + 1
    alt = torch.ones(n, device="cuda")
    alt[1::2] = -1.0
    assert device_sum(g, alt, n) == 1.0


def test_empty_sum_is_zero(g):
    out = torch.full((1,), 5.0, dtype=torch.float32, device="cuda")
    st = g.reduce_f32_sum(0, 0, out.data_ptr(), 0, torch.cuda.current_stream().cuda_stream)
    assert st == g.OK and out.item() == 0.0


def test_rerun_and_streams_bit_identical(g):
    n = 5_000_000
    x = synth.normal((n,), 78).reshape(-1)
    xd = torch.from_numpy(x).cuda()
    ref = device_sum(g, xd, n)
    outs = []
    streams = [torch.cuda.Stream() for _ in range(3)]
    for st in streams:
        with torch.cuda.stream(st):
            o = torch.empty(1, dtype=torch.float32, device="cuda")
            assert g.reduce_f32_sum(n, xd.data_ptr(), o.data_ptr(), 0, st.cuda_stream) == g.OK
            outs.append(o)
    torch.cuda.synchronize()
    assert all(o.item() == ref for o in outs)


def test_full_size_of_the_pages_measurement(g):
    # 2^26 fp32 values, the size "GPU compute shaders" times ("Complexity and
    # constants"), in the launch configuration the benchmark uses
    n = 1 << 26
    x = synth.uniform_pm1((n,), 1026).reshape(-1)
    xd = torch.from_numpy(x).cuda()
    got = device_sum(g, xd, n)
    s64, scale = oracle.vector_sum(x)
    assert abs(got - s64) <= bound(n, 0, scale)
    assert device_sum(g, xd, n) == got


def test_vector_sum_wrapper(g):
    x = torch.arange(1000, dtype=torch.float32, device="cuda")
    assert g.vector_sum(x).item() == 999 * 1000 / 2
    with pytest.raises(TypeError):
        g.vector_sum(x.view(10, 100))
