import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload")


@pytest.fixture(scope="session")
def golden_dir():
    return GOLDEN


@pytest.fixture(autouse=True)
def _debug_build_skips_nothing(request):
    """When the suite runs on the bounds-checked build (QNRE_LIB names
    libqnre_debug.so), every GPU test must end with no access skipped."""
    yield
    if "gpu" not in request.keywords or not os.environ.get("QNRE_LIB", "").endswith("libqnre_debug.so"):
        return
    from ulysses_qkv_proj_gb300 import binding as qb
    assert qb.debug_bounds(reset=True) == 0, "the debug build skipped out-of-range accesses"
