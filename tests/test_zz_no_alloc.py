"""The no-allocation forward, xhc_sublayer_fwd_noalloc.

It exists for callers that cannot allocate device memory (a hook running
inside another framework's memory pool, a C caller that only holds its input
and output buffers): instead of a caller workspace it uses scratch built into
the library.  These tests call it through the C ABI and check that it gives
the same result as xhc_sublayer_fwd with a caller workspace, on two calls in a
row with different inputs (the shared scratch must not leak one call's state
into the next), and that a call too large for the built-in scratch is refused
before anything runs.

This file is collected last on purpose, so that a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import xhc_oracle as xo
from residual_stream_expansion_xhc_b300 import inputs as xin
from tests.xhc_testlib import TOL, dev_act, dev_f32, host_f64, tdtype

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from residual_stream_expansion_xhc_b300 import _lib, api

CASES = [
    # (workload, keep the logits in `saved`)
    (xin.Workload("noalloc_bf16", 40, B=2, S=96, N=16, C=512, k=4, dtype="bf16"), False),
    (xin.Workload("noalloc_bf16_saved", 43, B=1, S=150, N=16, C=256, k=4, dtype="bf16"), True),
    (xin.Workload("noalloc_f32", 41, B=1, S=70, N=8, C=96, k=3, dtype="f32"), False),
    # fp32 with `saved` needs no scratch at all: the call goes straight through
    (xin.Workload("noalloc_f32_saved", 44, B=2, S=33, N=8, C=64, k=2, dtype="f32"), True),
]


def _run(wl, t, use_noalloc, keep_saved):
    sh = api.make_shape(wl.B, wl.S, wl.N, wl.C, wl.k, tdtype(wl), wl.iters, wl.eps)
    X = dev_act(wl, t.X)
    out = dev_act(wl, t.out)
    conv = tuple(dev_f32(w) for w in t.conv)
    W = dev_f32(t.W)
    x_in = torch.empty(wl.B, wl.S, wl.C, dtype=tdtype(wl), device="cuda")
    act = torch.empty(wl.B, wl.S, wl.k, wl.C, dtype=tdtype(wl), device="cuda")
    saved = torch.empty(wl.B, wl.S, wl.P + 1, device="cuda") if keep_saved else None
    if use_noalloc:
        api.xhc_sublayer_fwd_noalloc(sh, X, X, out, conv, W, t.idx, x_in=x_in, saved=saved, saved_active=act)
    else:
        ws = api.workspace(api.xhc_fwd_workspace_need(sh, keep_saved))
        api.xhc_sublayer_fwd(sh, X, X, out, conv, W, t.idx, x_in=x_in, saved=saved, saved_active=act, workspace=ws)
    torch.cuda.synchronize()
    api.xhc_device_status()
    res = {"X'": X, "x_in": x_in, "saved_active": act}
    if keep_saved:
        res["saved"] = saved
    return res


@pytest.mark.parametrize("wl,keep_saved", CASES, ids=[w.name for w, _ in CASES])
def test_noalloc_matches_workspace_path_twice(wl, keep_saved):
    if wl.dtype == "f32" and keep_saved:
        sh = api.make_shape(wl.B, wl.S, wl.N, wl.C, wl.k, tdtype(wl), wl.iters, wl.eps)
        assert api.xhc_fwd_workspace_need(sh, True) == 0
    for call in range(2):
        # a different seeded draw for each call
        t = xin.make(xin.scaled(wl, wid=wl.wid + 100 * call))
        ref = _run(wl, t, use_noalloc=False, keep_saved=keep_saved)
        got = _run(wl, t, use_noalloc=True, keep_saved=keep_saved)
        assert set(ref) == set(got)
        for key in ref:
            e = xo.max_rel_err(host_f64(got[key]), host_f64(ref[key]))
            assert e <= TOL[wl.dtype], f"call {call}, {key}: err {e}"


def test_noalloc_refuses_calls_beyond_its_scratch():
    # 100,000 bf16 tokens need 100,000 x (48 + 49) x 4 bytes > 32 MiB without
    # `saved`: refused before any launch; with `saved` (48 x 4 bytes per
    # token, plus the split copy of W) they fit
    sh = _lib.XhcShape(1, 100000, 16, 256, 4, _lib.XHC_BF16, 20, 1e-6)
    assert api.xhc_fwd_workspace_need(sh, False) > 32 << 20 >= api.xhc_fwd_workspace_need(sh, True)
    idx = (ctypes.c_int32 * 4)(0, 1, 2, 3)
    fake = ctypes.c_void_p(1 << 20)
    st = _lib.LIB.xhc_sublayer_fwd_noalloc(ctypes.byref(sh), fake, fake, fake, None, None, None, fake, idx, None,
                                           None, None, None)
    assert st == 5                     # XHC_ERR_WORKSPACE
