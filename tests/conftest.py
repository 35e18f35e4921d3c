import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running")


@pytest.fixture(scope="session")
def root():
    return ROOT


@pytest.fixture(autouse=True)
def _debug_build_record(request):
    """Under the debug build (XHC_DEBUG=1) every GPU test must leave no
    out-of-extent access recorded by the streaming kernels' bounds checks."""
    yield
    if os.environ.get("XHC_DEBUG") == "1" and request.node.get_closest_marker("gpu"):
        from residual_stream_expansion_xhc_b300 import api
        st, line, addr = api.xhc_debug_record()
        assert st == 0, f"out-of-extent access recorded at source line {line}, address {addr:#x}"
