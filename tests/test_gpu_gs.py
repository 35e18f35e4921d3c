"""GPU-vs-oracle parity of the fused sublayer forward and backward with
modified Gram-Schmidt of the TFA components, through the C ABI.

Method: "xHC: Expanded Hyper-Connections" (qingkeai.online), section
"Conv / Gram-Schmidt".  The GPU forms each token's Gram matrix of the raw
components and applies the Gram-Schmidt steps to coefficients; the oracle runs
the steps on the vectors in fp64.  The conv weights are drawn with std 0.3 so
that the components are of the size of `out` and correlated with it: each case
first checks that Gram-Schmidt moves the oracle's result by far more than the
tolerance, so that the parity check can tell the two apart.

Tolerance: the bf16 bound of the error measure max_i |g_i - r_i| /
max(|r_i|, rms(r)), 2e-2; inactive rows bit for bit.
"""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import xhc_oracle as xo
from residual_stream_expansion_xhc_b300 import inputs as xin
from tests.xhc_testlib import TOL, dev_act, dev_f32, host_f64, oracle_inputs, tdtype

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from residual_stream_expansion_xhc_b300 import api


def _wl(name, wid, **kw):
    base = dict(N=16, k=4, dtype="bf16", conv_std=0.3, gram_schmidt=True)
    base.update(kw)
    return xin.Workload(name, wid, **base)


CASES = {
    "gs_ragged": _wl("gs_ragged", 31, B=2, S=77, C=512),
    "gs_c2048": _wl("gs_c2048", 32, B=1, S=130, C=2048),
    "gs_s1": _wl("gs_s1", 33, B=3, S=1, C=256),
    "gs_s5": _wl("gs_s5", 34, B=2, S=5, C=256),
    "gs_s12": _wl("gs_s12", 35, B=2, S=12, C=256),
    "gs_k2": _wl("gs_k2", 36, B=2, S=40, N=6, k=2, C=256),
    "gs_zero_conv": _wl("gs_zero_conv", 37, B=1, S=33, C=256, conv="zero"),
}


def _shape(wl):
    return api.make_shape(wl.B, wl.S, wl.N, wl.C, wl.k, tdtype(wl), wl.iters, wl.eps, wl.gram_schmidt)


def _tensors(name, grads=False, dx_in=False):
    wl = CASES[name]
    t = xin.make(wl, grads=grads, dx_in=dx_in)
    if name == "gs_k2":
        # u_2 = u_1 exactly (the K = 8 taps repeat the K = 4 ones, then zeros):
        # a dependent component, whose projections are skipped
        w4, w8, w12 = t.conv
        w8 = np.concatenate([w4, np.zeros((wl.C, 4), np.float32)], axis=1)
        t.conv = (w4, w8, w12)
    return wl, t


def _fwd(wl, t):
    sh = _shape(wl)
    X = dev_act(wl, t.X)
    X0 = X.clone()
    out = dev_act(wl, t.out)
    conv = None if t.conv is None else tuple(dev_f32(w) for w in t.conv)
    W = dev_f32(t.W)
    x_in = torch.empty(wl.B, wl.S, wl.C, dtype=tdtype(wl), device="cuda")
    saved = torch.empty(wl.B, wl.S, wl.P + 1, dtype=torch.float32, device="cuda")
    act = torch.empty(wl.B, wl.S, wl.k, wl.C, dtype=tdtype(wl), device="cuda")
    ws = api.workspace(api.xhc_fwd_workspace_need(sh, True))
    api.xhc_sublayer_fwd(sh, X, X, out, conv, W, t.idx, x_in=x_in, saved=saved, saved_active=act, workspace=ws)
    torch.cuda.synchronize()
    api.xhc_device_status()
    return dict(X0=X0, Xp=X, x_in=x_in, saved=saved, act=act)


@pytest.mark.parametrize("name", list(CASES))
def test_gs_forward_parity(name):
    wl, t = _tensors(name)
    g = _fwd(wl, t)
    X, out, conv, W, idx = oracle_inputs(wl, t)
    ref = xo.forward(X, out, conv, W, idx, iters=wl.iters, eps=wl.eps, gs=True)
    tol = TOL[wl.dtype]
    idx = list(idx)
    inactive = [n for n in range(wl.N) if n not in idx]
    if conv is not None and name != "gs_zero_conv":
        plain = xo.forward(X, out, conv, W, idx, iters=wl.iters, eps=wl.eps)
        assert xo.max_rel_err(plain["Xp"][:, :, idx], ref["Xp"][:, :, idx]) > 5 * tol
    assert torch.equal(g["Xp"][:, :, inactive].view(torch.int16), g["X0"][:, :, inactive].view(torch.int16))
    e = xo.max_rel_err(host_f64(g["Xp"][:, :, idx]), ref["Xp"][:, :, idx])
    assert e <= tol, f"X' err {e}"
    e = xo.max_rel_err(host_f64(g["x_in"]), ref["x_in"])
    assert e <= tol, f"x_in err {e}"


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("mode", ["active+saved+dxin", "recompute", "no_dxin"])
def test_gs_backward_parity(name, mode):
    with_dxin = mode != "no_dxin"
    wl, t = _tensors(name, grads=True, dx_in=with_dxin)
    fw = _fwd(wl, t)
    sh = _shape(wl)
    out = dev_act(wl, t.out)
    conv = None if t.conv is None else tuple(dev_f32(w) for w in t.conv)
    W = dev_f32(t.W)
    dXp = dev_act(wl, t.dXp)
    dxi = dev_act(wl, t.dx_in) if with_dxin else None
    if mode == "recompute":
        X_state, act, saved = fw["X0"], None, None
    else:
        X_state, act, saved = fw["Xp"], fw["act"], fw["saved"]
    dX = torch.empty_like(dXp)
    dout = torch.empty_like(out)
    dconv = None if conv is None else tuple(torch.empty_like(w) for w in conv)
    dW = torch.empty_like(W)
    ws = api.workspace(api.xhc_bwd_workspace_bytes(sh))
    api.xhc_sublayer_bwd(sh, X_state, act, out, conv, W, t.idx, saved, dXp, dxi, dX, dout, dconv, dW, ws)
    torch.cuda.synchronize()
    api.xhc_device_status()
    X, out64, conv64, W64, idx = oracle_inputs(wl, t)
    dxi64 = xin.to_f64(wl, t.dx_in) if with_dxin else None
    ref = xo.backward(X, out64, conv64, W64, idx, xin.to_f64(wl, t.dXp), dxi64, iters=wl.iters, eps=wl.eps, gs=True)
    tol = TOL[wl.dtype]
    if conv64 is not None and name != "gs_zero_conv":
        plain = xo.backward(X, out64, conv64, W64, idx, xin.to_f64(wl, t.dXp), dxi64, iters=wl.iters, eps=wl.eps)
        assert xo.max_rel_err(plain["dout"], ref["dout"]) > 5 * tol
    for key, got in (("dX", dX), ("dout", dout), ("dW", dW)):
        e = xo.max_rel_err(host_f64(got), ref[key])
        assert e <= tol, f"{key} err {e}"
    for j in range(3):
        e = xo.max_rel_err(host_f64(dconv[j]), ref["dconv"][j])
        assert e <= tol, f"dw{(4, 8, 12)[j]} err {e}"


def test_gs_without_conv_is_plain_update():
    wl = dataclasses.replace(CASES["gs_ragged"], name="gs_noconv", conv="none")
    t = xin.make(wl)
    g = _fwd(wl, t)
    X, out, conv, W, idx = oracle_inputs(wl, t)
    ref = xo.forward(X, out, None, W, idx, iters=wl.iters, eps=wl.eps)
    e = xo.max_rel_err(host_f64(g["Xp"][:, :, list(idx)]), ref["Xp"][:, :, list(idx)])
    assert e <= TOL[wl.dtype]


def test_gs_bitwise_repeatable():
    wl, t = _tensors("gs_ragged")
    a = _fwd(wl, t)
    b = _fwd(wl, t)
    assert torch.equal(a["Xp"], b["Xp"])
