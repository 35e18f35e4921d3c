"""GPU-vs-oracle parity of the sublayer update with per-token active sets
chosen by the router (xhc_sublayer_fwd_routed), through the C ABI.

Method: "xHC: Expanded Hyper-Connections" (qingkeai.online), section "Dense
read, sparse write".  The GPU's scores and logits are compared with the
oracle's.  The GPU's active set of every token must be a valid router choice
for the oracle's logits (``check_selection``): the fixed streams first and in
order, the routed slots in descending logit order, every chosen routed logit
at least every unchosen one; both conditions within twice the largest
GPU-vs-oracle logit error of the case, so that a choice may differ from the
oracle's only where two logits tie to within that rounding.  Write-back and
dense read are then compared on every token against the oracle run with the
GPU's active sets: the bf16 bound 2e-2 of max_i |g_i - r_i| / max(|r_i|,
rms(r)); rows outside each token's active set bit for bit.
"""
import numpy as np
import pytest
import torch

from oracle import xhc_oracle as xo
from residual_stream_expansion_xhc_b300 import inputs as xin
from tests.xhc_testlib import TOL, check_selection, dev_act, dev_f32, host_f64, oracle_inputs, tdtype

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from residual_stream_expansion_xhc_b300 import api

CASES = {
    "router_ragged": (xin.Workload("router_ragged", 51, B=2, S=77, N=16, C=512, k=4, dtype="bf16", conv_std=0.3),
                      2),
    "router_c2048": (xin.Workload("router_c2048", 52, B=1, S=130, N=16, C=2048, k=4, dtype="bf16"), 2),
    "router_s5_nofixed": (xin.Workload("router_s5", 53, B=3, S=5, N=16, C=256, k=4, dtype="bf16"), 0),
    "router_k2": (xin.Workload("router_k2", 54, B=2, S=40, N=6, C=256, k=2, dtype="bf16"), 1),
    "router_noconv": (xin.Workload("router_noconv", 55, B=2, S=40, N=16, C=256, k=4, dtype="bf16", conv="none"), 2),
    "router_all_fixed": (xin.Workload("router_all_fixed", 56, B=1, S=33, N=16, C=256, k=4, dtype="bf16"), 4),
}


def _logit_tol(g, r_ref, N):
    """Twice the largest logit error of the GPU against the oracle (a swap is
    valid only where two oracle logits are closer than that), and that error."""
    err = float(np.abs(g["rrec"][..., N:2 * N] - r_ref).max())
    assert err < 1e-3, f"router logit error {err}"
    return 2.0 * err + 1e-6, err


def _router_weights(wl):
    # logits W_r . LN(v) with a standard deviation of about 1
    std = 1.0 / np.sqrt(wl.N * wl.C)
    return (np.random.default_rng(1000 * wl.wid + 77).standard_normal((wl.N, wl.N * wl.C)) * std).astype(np.float32)


def _run(wl, t, W_r, fixed):
    sh = api.make_shape(wl.B, wl.S, wl.N, wl.C, wl.k, tdtype(wl), wl.iters, wl.eps)
    X = dev_act(wl, t.X)
    X0 = X.clone()
    out = dev_act(wl, t.out)
    conv = None if t.conv is None else tuple(dev_f32(w) for w in t.conv)
    x_in = torch.empty(wl.B, wl.S, wl.C, dtype=tdtype(wl), device="cuda")
    saved = torch.empty(wl.B, wl.S, wl.P + 1, device="cuda")
    act = torch.empty(wl.B, wl.S, wl.k, wl.C, dtype=tdtype(wl), device="cuda")
    tok_idx = torch.empty(wl.B, wl.S, wl.k, dtype=torch.int32, device="cuda")
    rrec = torch.empty(wl.B, wl.S, 2 * wl.N + 2, device="cuda")
    ws = api.workspace(api.xhc_fwd_routed_workspace_bytes(sh))
    api.xhc_sublayer_fwd_routed(sh, X, X, out, conv, dev_f32(t.W), dev_f32(W_r), fixed, tok_idx, rrec, ws,
                                x_in=x_in, saved=saved, saved_active=act)
    torch.cuda.synchronize()
    api.xhc_device_status()
    rr = rrec.cpu().numpy().astype(np.float64)
    return dict(X0=X0, Xp=X, x_in=x_in, idx=tok_idx.cpu().numpy(), scores=rr[..., : wl.N], rrec=rr, act=act,
                tok_idx=tok_idx, rrec_dev=rrec, saved=saved)


@pytest.mark.parametrize("name", list(CASES))
def test_routed_forward_parity(name):
    wl, nf = CASES[name]
    t = xin.make(wl)
    W_r = _router_weights(wl)
    fixed = [int(a) for a in t.idx[:nf]]
    g = _run(wl, t, W_r, fixed)
    X, out, conv, W, _ = oracle_inputs(wl, t)
    W_r64 = W_r.astype(np.float64)
    r_ref = np.zeros((wl.B, wl.S, wl.N))
    s_ref = np.zeros((wl.B, wl.S, wl.N))
    # the record's scores, logits, LayerNorm mean and sd
    for b in range(wl.B):
        s_ref[b], r_ref[b], y, sd = xo.router_scores(X[b], W_r64, wl.eps)
        assert np.abs(g["rrec"][b, :, 2 * wl.N + 1] - sd).max() < 1e-4 * sd.max()
        mean = X[b].reshape(wl.S, -1).mean(axis=1)
        assert np.abs(g["rrec"][b, :, 2 * wl.N] - mean).max() < 1e-4
    assert np.abs(g["scores"] - s_ref).max() < 1e-4
    ltol, _ = _logit_tol(g, r_ref, wl.N)
    # the selection: a valid choice for every token
    check_selection(g["idx"], r_ref, fixed, wl.k, ltol)
    # the update with the GPU's active sets, every token
    ref = xo.forward_routed(X, out, conv, W, W_r64, fixed, wl.k, iters=wl.iters, eps=wl.eps, idx=g["idx"])
    tol = TOL[wl.dtype]
    Xp, X0 = host_f64(g["Xp"]), host_f64(g["X0"])
    inactive = np.ones((wl.B, wl.S, wl.N), dtype=bool)
    np.put_along_axis(inactive, g["idx"].astype(np.int64), False, axis=-1)
    assert np.array_equal(Xp[inactive], X0[inactive])
    err = xo.max_rel_err(Xp, ref["Xp"])
    assert err <= tol, f"X' err {err}"
    e = xo.max_rel_err(host_f64(g["x_in"]), ref["x_in"])
    assert e <= tol, f"x_in err {e}"
    # saved active rows: the slots' rows before the update, bit for bit
    act = g["act"].view(torch.int16).cpu().numpy()
    x0 = g["X0"].view(torch.int16).cpu().numpy()
    gidx = g["idx"].astype(np.int64)
    assert np.array_equal(act, np.take_along_axis(x0, gidx[..., None], axis=2))


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("with_dxin", [False, True])
@pytest.mark.parametrize("in_place", [False, True])
def test_routed_backward_parity(name, with_dxin, in_place):
    """in_place: the backward gets the state after the in-place forward and
    the saved active rows, and must leave the state before the update in it,
    bit for bit."""
    wl, nf = CASES[name]
    t = xin.make(wl, grads=True, dx_in=with_dxin)
    W_r = _router_weights(wl)
    fixed = [int(a) for a in t.idx[:nf]]
    g = _run(wl, t, W_r, fixed)
    sh = api.make_shape(wl.B, wl.S, wl.N, wl.C, wl.k, tdtype(wl), wl.iters, wl.eps)
    out = dev_act(wl, t.out)
    conv = None if t.conv is None else tuple(dev_f32(w) for w in t.conv)
    W, Wr = dev_f32(t.W), dev_f32(W_r)
    dXp = dev_act(wl, t.dXp)
    dxi = dev_act(wl, t.dx_in) if with_dxin else None
    dX = torch.empty_like(dXp)
    dout = torch.empty_like(out)
    dconv = None if conv is None else tuple(torch.empty_like(w) for w in conv)
    dW, dW_r = torch.empty_like(W), torch.empty_like(Wr)
    ws = api.workspace(api.xhc_bwd_routed_workspace_bytes(sh))
    state = g["Xp"] if in_place else g["X0"]
    api.xhc_sublayer_bwd_routed(sh, state, out, conv, W, Wr, fixed, g["saved"], g["tok_idx"], g["rrec_dev"], dXp,
                                dxi, dX, dout, dconv, dW, dW_r, ws, saved_active=g["act"] if in_place else None)
    torch.cuda.synchronize()
    api.xhc_device_status()
    if in_place:
        assert torch.equal(state.view(torch.int16), g["X0"].view(torch.int16))
    X, out64, conv64, W64, _ = oracle_inputs(wl, t)
    ref = xo.backward_routed(X, out64, conv64, W64, W_r.astype(np.float64), fixed, wl.k, xin.to_f64(wl, t.dXp),
                             xin.to_f64(wl, t.dx_in) if with_dxin else None, iters=wl.iters, eps=wl.eps,
                             idx=g["idx"])
    tol = TOL[wl.dtype]
    for key, got in (("dX", dX), ("dout", dout), ("dW", dW), ("dW_r", dW_r)):
        e = xo.max_rel_err(host_f64(got), ref[key])
        assert e <= tol, f"{key} err {e}"
    if conv is not None:
        for j in range(3):
            e = xo.max_rel_err(host_f64(dconv[j]), ref["dconv"][j])
            assert e <= tol, f"dw{(4, 8, 12)[j]} err {e}"


def test_routed_full_shape_one_sequence():
    """One sequence of the router workload at full width (S = 4096, C = 2048):
    forward and backward against the oracle on every token, with the GPU's
    active sets (their own check is the forward test's).  In place, as in
    training: the backward gets the updated state and the saved active rows
    and leaves the state before the update."""
    wl = xin.scaled(xin.WORKLOADS["router_bf16"], B=1)
    t = xin.make(wl, grads=True)
    W_r = t.extra["W_r"]
    fixed = [int(a) for a in t.idx[: wl.router_fixed]]
    g = _run(wl, t, W_r, fixed)
    X, out, conv, W, _ = oracle_inputs(wl, t)
    tol = TOL[wl.dtype]
    sh = api.make_shape(wl.B, wl.S, wl.N, wl.C, wl.k, tdtype(wl), wl.iters, wl.eps)
    conv_d = tuple(dev_f32(w) for w in t.conv)
    out_d, W_d, Wr_d, dXp = dev_act(wl, t.out), dev_f32(t.W), dev_f32(W_r), dev_act(wl, t.dXp)
    dX, dout = torch.empty_like(dXp), torch.empty_like(out_d)
    dconv = tuple(torch.empty_like(w) for w in conv_d)
    dW, dW_r = torch.empty_like(W_d), torch.empty_like(Wr_d)
    ws = api.workspace(api.xhc_bwd_routed_workspace_bytes(sh))
    Xp = host_f64(g["Xp"])
    api.xhc_sublayer_bwd_routed(sh, g["Xp"], out_d, conv_d, W_d, Wr_d, fixed, g["saved"], g["tok_idx"],
                                g["rrec_dev"], dXp, None, dX, dout, dconv, dW, dW_r, ws, saved_active=g["act"])
    torch.cuda.synchronize()
    api.xhc_device_status()
    assert torch.equal(g["Xp"].view(torch.int16), g["X0"].view(torch.int16))
    W_r64 = W_r.astype(np.float64)
    # forward: the routed update reproduced with the GPU's active sets
    ref_s, ref_r, _, _ = xo.router_scores(X[0], W_r64, wl.eps)
    assert np.abs(g["scores"][0] - ref_s).max() < 1e-4
    ltol, _ = _logit_tol(g, ref_r[None], wl.N)
    check_selection(g["idx"], ref_r[None], fixed, wl.k, ltol)
    fr = xo.forward_routed(X, out, conv, W, W_r64, fixed, wl.k, iters=wl.iters, eps=wl.eps, idx=g["idx"])
    X0 = host_f64(g["X0"])
    inactive = np.ones((wl.B, wl.S, wl.N), dtype=bool)
    np.put_along_axis(inactive, g["idx"].astype(np.int64), False, axis=-1)
    assert np.array_equal(Xp[inactive], X0[inactive])
    for key, got in (("Xp", Xp), ("x_in", host_f64(g["x_in"]))):
        e = xo.max_rel_err(got, fr[key])
        assert e <= tol, f"{key} err {e}"
    br = xo.backward_routed(X, out, conv, W, W_r64, fixed, wl.k, xin.to_f64(wl, t.dXp), None, iters=wl.iters,
                            eps=wl.eps, idx=g["idx"])
    for key, got in (("dX", dX), ("dout", dout), ("dW", dW), ("dW_r", dW_r)):
        e = xo.max_rel_err(host_f64(got), br[key])
        assert e <= tol, f"{key} err {e}"
    for j in range(3):
        e = xo.max_rel_err(host_f64(dconv[j]), br["dconv"][j])
        assert e <= tol, f"dw{(4, 8, 12)[j]} err {e}"
