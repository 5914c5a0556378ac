import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload cases")


@pytest.fixture(scope="session")
def lib():
    """The built C-ABI library on a GPU machine; GPU tests fail loudly when it is missing."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from ragged_grouped_gemm_device_gb300 import _lib
    return _lib.load()


@pytest.fixture(autouse=True)
def _debug_build_checks(request):
    """With MOE_GG_DEBUG_LIB=1 every GPU test runs on the debug build of the library; after each
    test the bounds checks of that build must all have held (a failure names the site, index and
    bound)."""
    yield
    import os
    if os.environ.get("MOE_GG_DEBUG_LIB") != "1" or request.node.get_closest_marker("gpu") is None:
        return
    from ragged_grouped_gemm_device_gb300 import _lib
    if _lib._lib is None:
        return
    assert _lib.moe_debug_build(), "MOE_GG_DEBUG_LIB=1, but the release build is the one loaded"
    mask, site, index, limit = _lib.moe_debug_report(reset=True)
    assert mask == 0, (f"debug build: bounds check failed at {_lib.moe_debug_site_name(site)} "
                       f"(index {index}, bound {limit}, site mask {mask:#x})")
