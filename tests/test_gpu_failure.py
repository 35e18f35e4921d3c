"""Failure detection on the GPU without a fault: the bounded device waits.

Every mbarrier wait of the tensor-core kernels gives up after a limit (2 s by
default, settable with xhc_set_wait_limit_ns), records XHC_ERR_TIMEOUT for
xhc_device_status and lets the kernel end; before it ends, each role waits
for the copies and tensor-core operations it issued.  The test shortens the
limit, makes the next coefficient projection issue none of its loads (its
consumers then wait on barriers that nothing completes, with nothing in
flight), and checks that the call ends after the short limit, that
xhc_device_status reports the timeout once and clears it, and that the next
normal call of the same entry point matches the oracle.
"""
import time

import numpy as np
import pytest
import torch

from oracle import xhc_oracle as xo
from residual_stream_expansion_xhc_b300 import inputs as xin
from tests.xhc_testlib import TOL, dev_act, dev_f32, host_f64, oracle_inputs, tdtype

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from residual_stream_expansion_xhc_b300 import _lib, api

XHC_OK, XHC_ERR_TIMEOUT = 0, 7
LIMIT_NS = 20_000_000          # 20 ms


def _fwd(wl, t, sh, X, ws):
    out = dev_act(wl, t.out)
    conv = tuple(dev_f32(w) for w in t.conv)
    x_in = torch.empty(wl.B, wl.S, wl.C, dtype=tdtype(wl), device="cuda")
    saved = torch.empty(wl.B, wl.S, wl.P + 1, device="cuda")
    api.xhc_sublayer_fwd(sh, X, X, out, conv, dev_f32(t.W), t.idx, x_in=x_in, saved=saved, workspace=ws)
    return x_in


def test_wait_runs_out_then_next_call_is_correct():
    wl = xin.Workload("wait_runout", 60, B=2, S=150, N=16, C=256, k=4, dtype="bf16")
    t = xin.make(wl)
    sh = api.make_shape(wl.B, wl.S, wl.N, wl.C, wl.k, tdtype(wl), wl.iters, wl.eps)
    ws = api.workspace(api.xhc_fwd_workspace_need(sh, True))
    torch.cuda.synchronize()
    assert _lib.LIB.xhc_device_status(None) == XHC_OK           # no earlier record
    try:
        api.xhc_set_wait_limit_ns(LIMIT_NS)
        api.xhc_debug_starve_next_projection()
        X = dev_act(wl, t.X)
        t0 = time.perf_counter()
        _fwd(wl, t, sh, X, ws)                                   # its outputs are undefined
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        assert _lib.LIB.xhc_device_status(None) == XHC_ERR_TIMEOUT
        assert _lib.LIB.xhc_device_status(None) == XHC_OK       # the record was cleared
        # the waits gave up after the short limit, not the default 2 s
        assert dt < 1.0, f"starved call took {dt:.3f} s"
    finally:
        api.xhc_set_wait_limit_ns(0)
    # the same entry point runs normally afterwards
    X = dev_act(wl, t.X)
    x_in = _fwd(wl, t, sh, X, ws)
    torch.cuda.synchronize()
    api.xhc_device_status()
    Xr, outr, convr, Wr, idx = oracle_inputs(wl, t)
    ref = xo.forward(Xr, outr, convr, Wr, idx, iters=wl.iters, eps=wl.eps)
    for name, got, want in (("X'", X, ref["Xp"]), ("x_in", x_in, ref["x_in"])):
        e = xo.max_rel_err(host_f64(got), want)
        assert e <= TOL[wl.dtype], f"{name} err {e}"
    inactive = [n for n in range(wl.N) if n not in list(idx)]
    np.testing.assert_array_equal(host_f64(X)[:, :, inactive], Xr[:, :, inactive])


def test_wait_limit_is_restored():
    """After the default limit is restored a normal call reports no timeout."""
    wl = xin.Workload("wait_default", 61, B=1, S=40, N=16, C=256, k=4, dtype="bf16")
    t = xin.make(wl)
    sh = api.make_shape(wl.B, wl.S, wl.N, wl.C, wl.k, tdtype(wl), wl.iters, wl.eps)
    ws = api.workspace(api.xhc_fwd_workspace_need(sh, True))
    api.xhc_set_wait_limit_ns(0)
    _fwd(wl, t, sh, dev_act(wl, t.X), ws)
    torch.cuda.synchronize()
    assert _lib.LIB.xhc_device_status(None) == XHC_OK
