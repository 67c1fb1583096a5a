import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes of host time)")


@pytest.fixture(scope="session")
def gemm_lib():
    """The built C-ABI library (compiled for sm_103a on first use)."""
    import dense_fp32_gemm_major_gb300 as g
    from dense_fp32_gemm_major_gb300 import _build

    _build.build_library()
    g.reload()
    return g


@pytest.fixture(scope="session")
def checked_lib(gemm_lib):
    """The index-checked build, libgemm_f32_checked.so (a ctypes handle with
    the same functions as the regular library)."""
    from dense_fp32_gemm_major_gb300 import _build

    _build.build_all()
    gemm_lib.reload()
    return gemm_lib.checked_library()
