"""Seeded synthetic workloads for the xHC sublayer update.

This module only draws random numbers and rounds them to the storage dtype; it
holds none of the update's arithmetic.  Both the CUDA path (tests, bench) and
the CPU oracle take their inputs from here, so that both see identical bits.

Seeds follow ``seed = 1000 * workload + 10 * sublayer + tensor`` with the
tensor codes below.  Values are drawn with numpy's PCG64 ``default_rng`` in
float32 and rounded to bf16 by round-to-nearest-even where the workload stores
bf16.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

T_X, T_OUT, T_W4, T_W8, T_W12, T_W, T_IDX, T_DXP, T_DXIN, T_WR = range(10)
CONV_KS = (4, 8, 12)


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shape, storage dtype and value distributions."""
    name: str
    wid: int                      # workload id used in the seed
    B: int
    S: int
    N: int
    C: int
    k: int
    dtype: str                    # "f32" or "bf16"
    layers: int = 1
    conv: str = "normal"          # "normal" | "zero" | "none"
    identity_idx: bool = False
    backward: bool = False
    w_std: float = 0.02
    conv_std: float = 0.02
    iters: int = 20
    eps: float = 1e-6
    gram_schmidt: bool = False    # orthogonalise the TFA components
    router_fixed: int = -1        # >= 0: router with this many fixed streams (W_r ~ N(0, 1/(N C)))

    @property
    def P(self) -> int:
        return self.N + 4 * self.k + self.k * self.k

    @property
    def tokens(self) -> int:
        return self.B * self.S

    @property
    def esize(self) -> int:
        return 4 if self.dtype == "f32" else 2


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", 1, B=1, S=256, N=16, C=256, k=4, dtype="f32"),
    "fwd_bf16": Workload("fwd_bf16", 2, B=4, S=4096, N=16, C=2048, k=4, dtype="bf16"),
    "stack8_bf16": Workload("stack8_bf16", 3, B=2, S=8192, N=16, C=4096, k=4, dtype="bf16", layers=8),
    "fwdbwd_bf16": Workload("fwdbwd_bf16", 4, B=4, S=4096, N=16, C=2048, k=4, dtype="bf16", backward=True),
    "mhc_bf16": Workload("mhc_bf16", 5, B=4, S=4096, N=4, C=2048, k=4, dtype="bf16",
                         conv="none", identity_idx=True, backward=True),
    # a quarter of the forward + backward workload (state 268 MB, above L2) for profiler captures
    "quarter_bf16": Workload("quarter_bf16", 6, B=1, S=4096, N=16, C=2048, k=4, dtype="bf16", backward=True),
    # forward + backward with Gram-Schmidt of the TFA components; conv weights
    # large enough (std 0.3) that the components are of the size of `out` and
    # correlated with it, so the orthogonalisation changes the write-back
    # the sublayer without TFA (u_0 = out only) at N = 16, k = 4
    "noconv_bf16": Workload("noconv_bf16", 8, B=4, S=4096, N=16, C=2048, k=4, dtype="bf16", conv="none",
                            backward=True),
    # per-token active sets from the router: the first two slots of the
    # layer's index list are fixed, two more are chosen per token
    "router_bf16": Workload("router_bf16", 9, B=4, S=4096, N=16, C=2048, k=4, dtype="bf16", backward=True,
                            router_fixed=2),
    "gs_bf16": Workload("gs_bf16", 7, B=4, S=4096, N=16, C=2048, k=4, dtype="bf16", backward=True,
                        conv_std=0.3, gram_schmidt=True),
    # a quarter of the router workload (state 268 MB, above L2) for profiler captures
    "router_quarter_bf16": Workload("router_quarter_bf16", 11, B=1, S=4096, N=16, C=2048, k=4, dtype="bf16",
                                    backward=True, router_fixed=2),
    # a two-sublayer stack at the eight-sublayer stack's width (state 537 MB,
    # above L2) for profiler captures of the fused stack step
    "stack2_quarter_bf16": Workload("stack2_quarter_bf16", 10, B=1, S=4096, N=16, C=4096, k=4, dtype="bf16",
                                    layers=2),
}


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    bias = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exactly equal float32 values."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def seed_of(wid: int, layer: int, tensor: int) -> int:
    return 1000 * wid + 10 * layer + tensor


def _normal(seed: int, shape, std: float = 1.0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


@dataclass
class Tensors:
    """Host copies of one sublayer's inputs.  Activations (X, out, dXp, dx_in)
    are held as storage-dtype arrays: float32 for f32 workloads, uint16 bf16
    bit patterns for bf16 workloads.  Weights are float32."""
    X: Optional[np.ndarray] = None
    out: Optional[np.ndarray] = None
    conv: Optional[tuple] = None
    W: Optional[np.ndarray] = None
    idx: Optional[np.ndarray] = None
    dXp: Optional[np.ndarray] = None
    dx_in: Optional[np.ndarray] = None
    extra: dict = field(default_factory=dict)


def _act(wl: Workload, seed: int, shape) -> np.ndarray:
    a = _normal(seed, shape)
    return a if wl.dtype == "f32" else bf16_bits(a)


def to_f64(wl: Workload, a: Optional[np.ndarray]) -> Optional[np.ndarray]:
    """Storage-dtype activation -> float64 values (exact)."""
    if a is None:
        return None
    if wl.dtype == "f32":
        return np.asarray(a, dtype=np.float64)
    return bf16_to_f32(a).astype(np.float64)


def active_idx(wl: Workload, layer: int) -> np.ndarray:
    if wl.identity_idx:
        return np.arange(wl.k, dtype=np.int32)
    rng = np.random.default_rng(seed_of(wl.wid, layer, T_IDX))
    return rng.permutation(wl.N)[: wl.k].astype(np.int32)


def make(wl: Workload, layer: int = 0, *, state: bool = True, grads: bool = False,
         dx_in: bool = False) -> Tensors:
    """Draw one sublayer's inputs.  ``state`` draws X (only layer 0 of a stack
    owns a fresh state), ``grads`` draws dX', ``dx_in`` draws dL/dx_in."""
    t = Tensors()
    B, S, N, C, k = wl.B, wl.S, wl.N, wl.C, wl.k
    if state:
        t.X = _act(wl, seed_of(wl.wid, layer, T_X), (B, S, N, C))
    t.out = _act(wl, seed_of(wl.wid, layer, T_OUT), (B, S, C))
    if wl.conv == "normal":
        t.conv = tuple(_normal(seed_of(wl.wid, layer, code), (C, K), wl.conv_std)
                       for code, K in zip((T_W4, T_W8, T_W12), CONV_KS))
    elif wl.conv == "zero":
        t.conv = tuple(np.zeros((C, K), np.float32) for K in CONV_KS)
    else:
        t.conv = None
    t.W = _normal(seed_of(wl.wid, layer, T_W), (wl.P, N * C), wl.w_std)
    t.idx = active_idx(wl, layer)
    if grads:
        t.dXp = _act(wl, seed_of(wl.wid, layer, T_DXP), (B, S, N, C))
    if dx_in:
        t.dx_in = _act(wl, seed_of(wl.wid, layer, T_DXIN), (B, S, C))
    if wl.router_fixed >= 0:
        # router logits W_r . LN(vec X) with a standard deviation of about 1
        t.extra["W_r"] = _normal(seed_of(wl.wid, layer, T_WR), (N, N * C), 1.0 / float(np.sqrt(N * C)))
    return t


def scaled(wl: Workload, **changes) -> Workload:
    """A copy of a workload with some fields changed (e.g. a smaller S for a
    parity case that the oracle finishes in seconds)."""
    d = dict(wl.__dict__)
    d.update(changes)
    return Workload(**d)
