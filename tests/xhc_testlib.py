"""Helpers shared by the GPU parity tests: device copies of seeded inputs,
the library calls for one sublayer, and the oracle on the same values."""
from __future__ import annotations

import numpy as np
import torch

from residual_stream_expansion_xhc_b300 import inputs as xin
from oracle import xhc_oracle as xo

TOL = {"f32": 1e-5, "bf16": 2e-2}


def dev_act(wl, a):
    """Storage-dtype host array -> device tensor of the workload dtype."""
    if a is None:
        return None
    if wl.dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
    return t.view(torch.bfloat16)


def dev_f32(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host_f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def tdtype(wl):
    return torch.float32 if wl.dtype == "f32" else torch.bfloat16


def oracle_inputs(wl, t):
    conv = None if t.conv is None else tuple(np.asarray(w, np.float64) for w in t.conv)
    return (xin.to_f64(wl, t.X), xin.to_f64(wl, t.out), conv, np.asarray(t.W, np.float64), t.idx)


def check_selection(gidx, r_ref, fixed, k, tol):
    """Every token's slots [B, S, k] are a valid choice for the logits r_ref
    [B, S, N] within tol; returns the fraction of tokens whose slots equal
    the oracle's own choice exactly."""
    B, S, N = r_ref.shape
    nf = len(fixed)
    gidx = np.asarray(gidx, dtype=np.int64)
    assert gidx.shape == (B, S, k)
    assert (gidx[..., :nf] == np.asarray(fixed, dtype=np.int64)).all(), "fixed slots"
    assert ((gidx >= 0) & (gidx < N)).all(), "slot out of range"
    srt = np.sort(gidx, axis=-1)
    assert (np.diff(srt, axis=-1) != 0).all(), "repeated stream"
    if nf == k:
        return float((gidx == np.asarray(fixed)).all(axis=-1).mean())
    routed = gidx[..., nf:]
    rr = np.take_along_axis(r_ref, routed, axis=-1)
    assert (np.diff(rr, axis=-1) <= tol).all(), "routed slots not in descending logit order"
    unchosen = np.ones((B, S, N), dtype=bool)
    np.put_along_axis(unchosen, gidx, False, axis=-1)
    if unchosen.any(axis=-1).all():
        best_left = np.where(unchosen, r_ref, -np.inf).max(axis=-1)
        assert (rr.min(axis=-1) >= best_left - tol).all(), "an unchosen stream outranks a chosen one"
    s_ref = 1.0 / (1.0 + np.exp(-r_ref))
    own = np.stack([xo.route(s_ref[b], fixed, k) for b in range(B)])
    return float((own == gidx).all(axis=-1).mean())
