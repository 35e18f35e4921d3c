"""GPU-vs-oracle parity of every entry point, through the C ABI.

Error measure: max_i |g_i - r_i| / max(|r_i|, rms(r)) per output tensor;
bounds 1e-5 (fp32 state) and 2e-2 (bf16 state, fp32 accumulation).  Index
handling is exact: the inactive streams of X' must equal the input bit for bit.
Sources: "xHC: Expanded Hyper-Connections" (qingkeai.online), sections
"Scaling N", "Temporal Feature Augmentation", "Dense read, sparse write".
"""
import numpy as np
import pytest
import torch

from residual_stream_expansion_xhc_b300 import inputs as xin
from oracle import xhc_oracle as xo
from tests.xhc_testlib import TOL, dev_act, dev_f32, host_f64, oracle_inputs, tdtype

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from residual_stream_expansion_xhc_b300 import api

# parity cases: small enough for the oracle, several tiles, a ragged tail
CASES = {
    "tiny_f32": xin.WORKLOADS["tiny_f32"],
    "bf16_ragged": xin.Workload("bf16_ragged", 11, B=2, S=77, N=16, C=512, k=4, dtype="bf16"),
    "bf16_c2048": xin.Workload("bf16_c2048", 12, B=1, S=130, N=16, C=2048, k=4, dtype="bf16"),
    "f32_ragged": xin.Workload("f32_ragged", 13, B=3, S=45, N=8, C=96, k=3, dtype="f32"),
    "mhc_bf16_small": xin.Workload("mhc_bf16_small", 14, B=2, S=70, N=4, C=256, k=4, dtype="bf16",
                                   conv="none", identity_idx=True),
    "bf16_odd_c": xin.Workload("bf16_odd_c", 15, B=1, S=33, N=6, C=72, k=2, dtype="bf16"),
    # degenerate lengths: one token, shorter than the longest convolution, exactly its length
    "bf16_s1": xin.Workload("bf16_s1", 16, B=3, S=1, N=16, C=256, k=4, dtype="bf16"),
    "bf16_s5": xin.Workload("bf16_s5", 17, B=2, S=5, N=16, C=256, k=4, dtype="bf16"),
    "bf16_s12": xin.Workload("bf16_s12", 18, B=2, S=12, N=16, C=256, k=4, dtype="bf16"),
    # fewest streams: one active of two
    "bf16_n2k1": xin.Workload("bf16_n2k1", 19, B=2, S=40, N=2, C=256, k=1, dtype="bf16"),
    # the sublayer without TFA (u_0 = out only) at N = 16, k = 4
    "bf16_noconv16": xin.Workload("bf16_noconv16", 21, B=2, S=77, N=16, C=512, k=4, dtype="bf16", conv="none"),
}


def shape_of(wl):
    return api.make_shape(wl.B, wl.S, wl.N, wl.C, wl.k, tdtype(wl), wl.iters, wl.eps)


def run_fwd(wl, t, inplace=True, want_x_in=True, want_saved=True, want_active=True):
    sh = shape_of(wl)
    X = dev_act(wl, t.X)
    X0 = X.clone()
    out = dev_act(wl, t.out)
    conv = None if t.conv is None else tuple(dev_f32(w) for w in t.conv)
    W = dev_f32(t.W)
    x_in = torch.empty(wl.B, wl.S, wl.C, dtype=tdtype(wl), device="cuda") if want_x_in else None
    saved = torch.empty(wl.B, wl.S, wl.P + 1, dtype=torch.float32, device="cuda") if want_saved else None
    act = torch.empty(wl.B, wl.S, wl.k, wl.C, dtype=tdtype(wl), device="cuda") if want_active else None
    need = api.xhc_fwd_workspace_need(sh, want_saved)
    ws = api.workspace(need) if need else None
    Xo = X if inplace else torch.full_like(X, float("nan"))
    api.xhc_sublayer_fwd(sh, X, Xo, out, conv, W, t.idx, x_in=x_in, saved=saved, saved_active=act, workspace=ws)
    torch.cuda.synchronize()
    return dict(X0=X0, Xp=Xo, x_in=x_in, saved=saved, act=act)


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("inplace", [True, False])
def test_sublayer_fwd_parity(name, inplace):
    wl = CASES[name]
    t = xin.make(wl)
    g = run_fwd(wl, t, inplace=inplace)
    ref = xo.forward(*oracle_inputs(wl, t), iters=wl.iters, eps=wl.eps)
    tol = TOL[wl.dtype]
    idx = list(t.idx)
    inactive = [n for n in range(wl.N) if n not in idx]
    Xp = g["Xp"]
    # index handling exact: inactive rows bit-identical to the input
    assert torch.equal(Xp[:, :, inactive].view(torch.int16 if wl.dtype == "bf16" else torch.int32),
                       g["X0"][:, :, inactive].view(torch.int16 if wl.dtype == "bf16" else torch.int32))
    e = xo.max_rel_err(host_f64(Xp[:, :, idx]), ref["Xp"][:, :, idx])
    assert e <= tol, f"X' active rows err {e}"
    e = xo.max_rel_err(host_f64(g["x_in"]), ref["x_in"])
    assert e <= tol, f"x_in err {e}"
    sv = host_f64(g["saved"])
    e = xo.max_rel_err(sv[..., : wl.P], ref["z"])
    assert e <= tol, f"z err {e}"
    e = xo.max_rel_err(sv[..., wl.P], ref["rstd"])
    assert e <= tol, f"rstd err {e}"
    # saved_active: the active rows before the update, bit for bit
    assert torch.equal(g["act"], g["X0"][:, :, idx])


@pytest.mark.parametrize("name", ["bf16_ragged", "tiny_f32"])
def test_sublayer_fwd_workspace_path(name):
    wl = CASES[name]
    t = xin.make(wl)
    a = run_fwd(wl, t, want_saved=True)
    b = run_fwd(wl, t, want_saved=False, want_x_in=False, want_active=False)
    assert torch.equal(a["Xp"], b["Xp"])


@pytest.mark.parametrize("name", list(CASES))
def test_coeffs_parity(name):
    wl = CASES[name]
    t = xin.make(wl)
    sh = shape_of(wl)
    X = dev_act(wl, t.X)
    W = dev_f32(t.W)
    B, S, N, k = wl.B, wl.S, wl.N, wl.k
    hpre = torch.empty(B, S, N, device="cuda")
    hpost = torch.empty(B, S, k, 4, device="cuda")
    hres = torch.empty(B, S, k, k, device="cuda")
    saved = torch.empty(B, S, wl.P + 1, device="cuda")
    x_in = torch.empty(B, S, wl.C, dtype=tdtype(wl), device="cuda")
    api.xhc_coeffs(sh, X, W, hpre, hpost, hres, saved, x_in)
    torch.cuda.synchronize()
    ref = xo.forward(*oracle_inputs(wl, t), iters=wl.iters, eps=wl.eps)
    tol = TOL[wl.dtype]
    for key, got in (("hpre", hpre), ("hpost", hpost), ("hres", hres), ("x_in", x_in)):
        e = xo.max_rel_err(host_f64(got), ref[key])
        assert e <= tol, f"{key} err {e}"
    # H^res columns sum to 1 (the last normalised axis)
    cs = hres.sum(dim=-2)
    assert (cs - 1).abs().max().item() < (1e-6 if wl.dtype == "f32" else 1e-5)


@pytest.mark.parametrize("name", ["tiny_f32", "bf16_ragged", "bf16_odd_c"])
def test_tfa_parity(name):
    wl = CASES[name]
    t = xin.make(wl)
    sh = shape_of(wl)
    out = dev_act(wl, t.out)
    conv = tuple(dev_f32(w) for w in t.conv)
    u = torch.empty(3, wl.B, wl.S, wl.C, dtype=tdtype(wl), device="cuda")
    api.xhc_tfa(sh, out, conv, u)
    torch.cuda.synchronize()
    ref_u = xo.tfa_components
    for b in range(wl.B):
        r = ref_u(xin.to_f64(wl, t.out)[b], tuple(np.asarray(w, np.float64) for w in t.conv))
        for j in range(3):
            e = xo.max_rel_err(host_f64(u[j, b]), r[j + 1])
            assert e <= TOL[wl.dtype], f"u{j + 1} err {e}"


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("inplace", [True, False])
def test_sparse_update_parity(name, inplace):
    """xhc_sparse_update with the oracle's coefficients (rounded to fp32) as
    inputs checks the write on its own."""
    wl = CASES[name]
    t = xin.make(wl)
    ref = xo.forward(*oracle_inputs(wl, t), iters=wl.iters, eps=wl.eps)
    sh = shape_of(wl)
    X = dev_act(wl, t.X)
    X0 = X.clone()
    out = dev_act(wl, t.out)
    conv = None if t.conv is None else tuple(dev_f32(w) for w in t.conv)
    hpost = dev_f32(ref["hpost"])
    hres = dev_f32(ref["hres"])
    Xo = X if inplace else torch.zeros_like(X)
    api.xhc_sparse_update(sh, X, Xo, out, conv, hpost, hres, t.idx)
    torch.cuda.synchronize()
    idx = list(t.idx)
    inactive = [n for n in range(wl.N) if n not in idx]
    assert torch.equal(Xo[:, :, inactive], X0[:, :, inactive])
    e = xo.max_rel_err(host_f64(Xo[:, :, idx]), ref["Xp"][:, :, idx])
    assert e <= TOL[wl.dtype], f"err {e}"


def run_bwd(wl, t, use_saved=True, use_active=True, dx_in=True, dX_alias=False):
    sh = shape_of(wl)
    fw = run_fwd(wl, t, inplace=True, want_saved=True, want_active=True)
    out = dev_act(wl, t.out)
    conv = None if t.conv is None else tuple(dev_f32(w) for w in t.conv)
    W = dev_f32(t.W)
    dXp = dev_act(wl, t.dXp)
    dxi = dev_act(wl, t.dx_in) if dx_in else None
    if use_active:
        X_state, act = fw["Xp"], fw["act"]
    else:
        X_state, act = fw["X0"], None
    saved = fw["saved"] if use_saved else None
    dX = dXp.clone() if dX_alias else torch.empty_like(dXp)
    dXp_arg = dX if dX_alias else dXp
    dout = torch.empty_like(out)
    dconv = None if conv is None else tuple(torch.empty_like(w) for w in conv)
    dW = torch.empty_like(W)
    ws = api.workspace(api.xhc_bwd_workspace_bytes(sh))
    api.xhc_sublayer_bwd(sh, X_state, act, out, conv, W, t.idx, saved, dXp_arg, dxi, dX, dout, dconv, dW, ws)
    torch.cuda.synchronize()
    return dict(dX=dX, dout=dout, dconv=dconv, dW=dW)


BWD_CASES = ["tiny_f32", "bf16_ragged", "f32_ragged", "mhc_bf16_small", "bf16_c2048", "bf16_odd_c", "bf16_s1",
             "bf16_s5", "bf16_s12", "bf16_n2k1", "bf16_noconv16"]


@pytest.mark.parametrize("name", BWD_CASES)
@pytest.mark.parametrize("mode", ["active+saved+dxin", "recompute", "no_dxin"])
def test_sublayer_bwd_parity(name, mode):
    wl = CASES[name]
    with_dxin = mode != "no_dxin"
    t = xin.make(wl, grads=True, dx_in=with_dxin)
    if mode == "active+saved+dxin":
        g = run_bwd(wl, t, use_saved=True, use_active=True, dx_in=True)
    elif mode == "recompute":
        g = run_bwd(wl, t, use_saved=False, use_active=False, dx_in=True)
    else:
        g = run_bwd(wl, t, use_saved=True, use_active=True, dx_in=False)
    X, out, conv, W, idx = oracle_inputs(wl, t)
    ref = xo.backward(X, out, conv, W, idx, xin.to_f64(wl, t.dXp), xin.to_f64(wl, t.dx_in) if with_dxin else None,
                      iters=wl.iters, eps=wl.eps)
    tol = TOL[wl.dtype]
    for key in ("dX", "dout", "dW"):
        e = xo.max_rel_err(host_f64(g[key]), ref[key])
        assert e <= tol, f"{key} err {e}"
    if conv is not None:
        for j in range(3):
            e = xo.max_rel_err(host_f64(g["dconv"][j]), ref["dconv"][j])
            assert e <= tol, f"dw{j} err {e}"


def test_bitwise_repeatable():
    wl = CASES["bf16_ragged"]
    t = xin.make(wl, grads=True, dx_in=True)
    a = run_bwd(wl, t)
    b = run_bwd(wl, t)
    for key in ("dX", "dout", "dW"):
        assert torch.equal(a[key], b[key])
    for x, y in zip(a["dconv"], b["dconv"]):
        assert torch.equal(x, y)


def test_empty_batch_is_noop():
    wl = xin.Workload("empty", 20, B=0, S=16, N=16, C=256, k=4, dtype="bf16")
    sh = shape_of(wl)
    W = torch.randn(wl.P, wl.N * wl.C, device="cuda")
    X = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    api.xhc_sublayer_fwd(sh, X, X, X, None, W, [0, 1, 2, 3])
    dW = torch.full_like(W, 7.0)
    ws = api.workspace(16)
    dX = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    api.xhc_sublayer_bwd(sh, X, None, X, None, W, [0, 1, 2, 3], None, X, None, dX, X, None, dW, ws)
    torch.cuda.synchronize()
    assert not dW.any()


def test_copy_kernel():
    a = torch.randn(1 << 20, device="cuda")
    b = torch.empty_like(a)
    api.xhc_copy(a, b)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
