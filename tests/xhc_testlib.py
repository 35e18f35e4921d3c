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
