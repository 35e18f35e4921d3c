"""The debug build (libxhc_debug.so, compiled with -DXHC_DEBUG).

Its forward update and backward column pass check every global load and
store against the extents of their launch's buffers; an access outside all of
them is skipped and recorded instead of faulting.  These tests run in child
processes that load the debug build (XHC_DEBUG=1):

- the checker's self-test: one checked load outside the registered extent
  (but inside the allocation) is skipped and recorded with its address;
- the GPU parity suites of the plain and the routed update, whose every test
  must also leave no record (the autouse fixture in conftest.py).
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SELFTEST = """
import torch
from residual_stream_expansion_xhc_b300 import _lib, api
assert _lib.DEBUG and _lib.LIB_PATH.endswith("libxhc_debug.so")
buf = torch.arange(64, dtype=torch.float32, device="cuda") + 1.0
out = torch.full((4,), -1.0, device="cuda")
assert api.xhc_debug_record()[0] == 0
api.xhc_debug_selftest(buf, out)
st, line, addr = api.xhc_debug_record()
assert st == 1 and line > 0, (st, line)
assert addr == buf.data_ptr() + 128, (hex(addr), hex(buf.data_ptr()))
assert float(out[0]) == 0.0                     # the load was skipped
assert api.xhc_debug_record()[0] == 0           # and the record cleared
print("selftest ok")
"""


def _child(args, timeout):
    env = dict(os.environ, XHC_DEBUG="1")
    return subprocess.run([sys.executable, *args], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=timeout)


def test_checker_records_and_skips_an_out_of_extent_load():
    r = _child(["-c", SELFTEST], 300)
    assert r.returncode == 0 and "selftest ok" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]


def test_parity_suites_leave_no_record_under_the_debug_build():
    r = _child(["-m", "pytest", "tests/test_gpu_parity.py", "tests/test_gpu_router.py", "-m", "gpu", "-x", "-q",
                "-p", "no:cacheprovider"], 1500)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
