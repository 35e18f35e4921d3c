"""GPU parity of the variant with H^res logits from the k active rows only.

Method: "xHC: Expanded Hyper-Connections" (qingkeai.online), section "Dense
read, sparse write": only the active streams take part in the residual mixing,
so its logits can come from their k*C state entries (the O(k^3 C) reading).
The library builds the full projection from W_pp and W_ra
(xhc_hres_active_weights) and reads dW_ra back from the full gradient
(xhc_hres_active_grad); both are compared bit for bit with the oracle's
mapping, and the fused forward and backward with the oracle's definition.
Tolerance: the bf16 bound 2e-2 of max_i |g_i - r_i| / max(|r_i|, rms(r)).
"""
import numpy as np
import pytest
import torch

from oracle import xhc_oracle as xo
from residual_stream_expansion_xhc_b300 import inputs as xin
from tests.xhc_testlib import TOL, dev_act, dev_f32, host_f64, tdtype

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from residual_stream_expansion_xhc_b300 import api

WL = xin.Workload("hres_active", 41, B=2, S=77, N=16, C=512, k=4, dtype="bf16")


def _weights(wl):
    rng = np.random.default_rng(4100)
    W_pp = (rng.standard_normal((wl.N + 4 * wl.k, wl.N * wl.C)) * 0.02).astype(np.float32)
    W_ra = (rng.standard_normal((wl.k * wl.k, wl.k * wl.C)) * 0.05).astype(np.float32)
    return W_pp, W_ra


def _shape(wl):
    return api.make_shape(wl.B, wl.S, wl.N, wl.C, wl.k, tdtype(wl), wl.iters, wl.eps)


def test_hres_active_weight_layout_and_gradient_gather():
    wl = WL
    t = xin.make(wl)
    W_pp, W_ra = _weights(wl)
    sh = _shape(wl)
    W = torch.empty(wl.P, wl.N * wl.C, device="cuda")
    api.xhc_hres_active_weights(sh, dev_f32(W_pp), dev_f32(W_ra), t.idx, W)
    dW = torch.randn(wl.P, wl.N * wl.C, device="cuda")
    dW_ra = torch.empty(wl.k * wl.k, wl.k * wl.C, device="cuda")
    api.xhc_hres_active_grad(sh, dW, t.idx, dW_ra)
    torch.cuda.synchronize()
    ref = xo.expand_hres_active(W_pp.astype(np.float64), W_ra.astype(np.float64), t.idx, wl.N, wl.C)
    assert np.array_equal(W.cpu().numpy().astype(np.float64), ref)
    assert np.array_equal(dW_ra.cpu().numpy(), xo.gather_hres_active(dW.cpu().numpy(), t.idx, wl.N, wl.C))


def test_hres_active_sublayer_parity():
    wl = WL
    t = xin.make(wl, grads=True)
    W_pp, W_ra = _weights(wl)
    sh = _shape(wl)
    W = torch.empty(wl.P, wl.N * wl.C, device="cuda")
    api.xhc_hres_active_weights(sh, dev_f32(W_pp), dev_f32(W_ra), t.idx, W)
    X = dev_act(wl, t.X)
    out = dev_act(wl, t.out)
    conv = tuple(dev_f32(w) for w in t.conv)
    saved = torch.empty(wl.B, wl.S, wl.P + 1, device="cuda")
    act = torch.empty(wl.B, wl.S, wl.k, wl.C, dtype=tdtype(wl), device="cuda")
    ws = api.workspace(api.xhc_fwd_workspace_need(sh, True))
    api.xhc_sublayer_fwd(sh, X, X, out, conv, W, t.idx, saved=saved, saved_active=act, workspace=ws)
    dX = torch.empty_like(X)
    dout = torch.empty_like(out)
    dconv = tuple(torch.empty_like(w) for w in conv)
    dW = torch.empty_like(W)
    bws = api.workspace(api.xhc_bwd_workspace_bytes(sh))
    api.xhc_sublayer_bwd(sh, X, act, out, conv, W, t.idx, saved, dev_act(wl, t.dXp), None, dX, dout, dconv, dW, bws)
    dW_ra = torch.empty(wl.k * wl.k, wl.k * wl.C, device="cuda")
    api.xhc_hres_active_grad(sh, dW, t.idx, dW_ra)
    torch.cuda.synchronize()
    api.xhc_device_status()
    X64, out64 = xin.to_f64(wl, t.X), xin.to_f64(wl, t.out)
    conv64 = tuple(np.asarray(w, np.float64) for w in t.conv)
    Wf = xo.expand_hres_active(W_pp.astype(np.float64), W_ra.astype(np.float64), t.idx, wl.N, wl.C)
    fr = xo.forward(X64, out64, conv64, Wf, t.idx, iters=wl.iters, eps=wl.eps)
    br = xo.backward(X64, out64, conv64, Wf, t.idx, xin.to_f64(wl, t.dXp), None, iters=wl.iters, eps=wl.eps)
    tol = TOL[wl.dtype]
    idx = list(t.idx)
    checks = [("X'", X[:, :, idx], fr["Xp"][:, :, idx]), ("z", saved[..., : wl.P], fr["z"]),
              ("dX", dX, br["dX"]), ("dout", dout, br["dout"]),
              ("dW_ra", dW_ra, xo.gather_hres_active(br["dW"], t.idx, wl.N, wl.C)),
              ("dW_pp", dW[: wl.N + 4 * wl.k], br["dW"][: wl.N + 4 * wl.k])]
    for name, got, ref in checks:
        e = xo.max_rel_err(host_f64(got), ref)
        assert e <= tol, f"{name} err {e}"
