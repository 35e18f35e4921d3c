"""Python binding of the xHC C ABI (include/xhc.h), same entry-point names.

Argument marshalling only: torch tensors are passed as device pointers with
the current CUDA stream (or an explicit one); the library's kernels do all of
the work.  Conventions (layouts, dtypes, ownership, errors) are those of the
C header; a non-zero status raises ``XhcError``.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import torch

from ._lib import LIB, XHC_BF16, XHC_F32, XhcError, XhcShape

Tensor = torch.Tensor
_DT = {torch.float32: XHC_F32, torch.bfloat16: XHC_BF16}


def make_shape(B: int, S: int, N: int, C: int, k: int, dtype, iters: int = 20, eps: float = 1e-6,
               gram_schmidt: bool = False) -> XhcShape:
    """Build an ``xhc_shape_t``; ``dtype`` is a torch dtype or "f32"/"bf16";
    ``gram_schmidt`` orthogonalises the TFA components in the fused sublayer
    forward and backward."""
    if isinstance(dtype, str):
        dt = {"f32": XHC_F32, "bf16": XHC_BF16}[dtype]
    else:
        dt = _DT[dtype]
    return XhcShape(B, S, N, C, k, dt, iters, eps, 1 if gram_schmidt else 0)


def num_logits(sh: XhcShape) -> int:
    return LIB.xhc_num_logits(ctypes.byref(sh))


def _p(t: Optional[Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _s(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _idx(idx: Sequence[int]):
    arr = (ctypes.c_int32 * len(idx))(*[int(i) for i in idx])
    return arr


def _conv(conv):
    if conv is None:
        return None, None, None
    return tuple(_p(w) for w in conv)


def _check(name: str, status: int):
    if status != 0:
        raise XhcError(name, status, LIB)


def xhc_coeffs(sh, X, W, hpre, hpost, hres, saved=None, x_in=None, stream=None):
    _check("xhc_coeffs", LIB.xhc_coeffs(ctypes.byref(sh), _p(X), _p(W), _p(hpre), _p(hpost), _p(hres),
                                        _p(saved), _p(x_in), _s(stream)))


def xhc_tfa(sh, out, conv, u, stream=None):
    w4, w8, w12 = _conv(conv)
    _check("xhc_tfa", LIB.xhc_tfa(ctypes.byref(sh), _p(out), w4, w8, w12, _p(u), _s(stream)))


def xhc_sparse_update(sh, X_in, X_out, out, conv, hpost, hres, idx, stream=None):
    w4, w8, w12 = _conv(conv)
    _check("xhc_sparse_update", LIB.xhc_sparse_update(ctypes.byref(sh), _p(X_in), _p(X_out), _p(out), w4, w8,
                                                      w12, _p(hpost), _p(hres), _idx(idx), _s(stream)))


def xhc_device_status(stream=None):
    """Raise if a bounded device-side wait gave up since the last check."""
    _check("xhc_device_status", LIB.xhc_device_status(_s(stream)))


def xhc_set_wait_limit_ns(ns: int):
    """Limit of the bounded device-side waits for later launches (0: 2 s)."""
    _check("xhc_set_wait_limit_ns", LIB.xhc_set_wait_limit_ns(ctypes.c_ulonglong(int(ns))))


def xhc_debug_starve_next_projection():
    """Test hook: the next coefficient projection issues no loads."""
    _check("xhc_debug_starve_next_projection", LIB.xhc_debug_starve_next_projection())


def xhc_debug_record():
    """(status, source line, address) of the debug build's first recorded
    out-of-extent access; status 1 = recorded (then cleared), 0 = none, -1 =
    release build."""
    line, addr = ctypes.c_ulonglong(0), ctypes.c_ulonglong(0)
    st = LIB.xhc_debug_record(ctypes.byref(line), ctypes.byref(addr))
    if st < -1:
        raise XhcError("xhc_debug_record", 6, LIB)
    return st, line.value, addr.value


def xhc_debug_selftest(buf, out, stream=None):
    _check("xhc_debug_selftest", LIB.xhc_debug_selftest(_p(buf), _p(out), _s(stream)))


def xhc_fwd_workspace_bytes(sh) -> int:
    return int(LIB.xhc_fwd_workspace_bytes(ctypes.byref(sh)))


def xhc_fwd_workspace_need(sh, keeps_saved: bool) -> int:
    return int(LIB.xhc_fwd_workspace_need(ctypes.byref(sh), 1 if keeps_saved else 0))


def xhc_bwd_workspace_bytes(sh) -> int:
    return int(LIB.xhc_bwd_workspace_bytes(ctypes.byref(sh)))


def xhc_sublayer_fwd(sh, X_in, X_out, out, conv, W, idx, x_in=None, saved=None, saved_active=None,
                     workspace=None, stream=None):
    w4, w8, w12 = _conv(conv)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("xhc_sublayer_fwd", LIB.xhc_sublayer_fwd(ctypes.byref(sh), _p(X_in), _p(X_out), _p(out), w4, w8, w12,
                                                    _p(W), _idx(idx), _p(x_in), _p(saved), _p(saved_active),
                                                    _p(workspace), ws_bytes, _s(stream)))


def xhc_sublayer_fwd_noalloc(sh, X_in, X_out, out, conv, W, idx, x_in=None, saved=None, saved_active=None,
                             stream=None):
    """xhc_sublayer_fwd without a workspace: for callers that may not allocate
    device memory.  Uses the library's built-in 32 MiB scratch (see the C
    header for the token limit and the rule that overlapping calls race)."""
    w4, w8, w12 = _conv(conv)
    _check("xhc_sublayer_fwd_noalloc",
           LIB.xhc_sublayer_fwd_noalloc(ctypes.byref(sh), _p(X_in), _p(X_out), _p(out), w4, w8, w12, _p(W),
                                        _idx(idx), _p(x_in), _p(saved), _p(saved_active), _s(stream)))


def xhc_sublayer_bwd(sh, X_state, saved_active, out, conv, W, idx, saved, dXp, dx_in, dX, dout, dconv, dW,
                     workspace, stream=None):
    w4, w8, w12 = _conv(conv)
    d4, d8, d12 = _conv(dconv)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("xhc_sublayer_bwd", LIB.xhc_sublayer_bwd(ctypes.byref(sh), _p(X_state), _p(saved_active), _p(out), w4,
                                                    w8, w12, _p(W), _idx(idx), _p(saved), _p(dXp), _p(dx_in),
                                                    _p(dX), _p(dout), d4, d8, d12, _p(dW), _p(workspace),
                                                    ws_bytes, _s(stream)))


def xhc_stack_fwd_workspace_bytes(sh) -> int:
    return LIB.xhc_stack_fwd_workspace_bytes(ctypes.byref(sh))


def _ptr_array(ts):
    """Host array of device pointers (None entries -> NULL), or NULL for None."""
    if ts is None:
        return None
    return (ctypes.c_void_p * len(ts))(*[None if t is None else t.data_ptr() for t in ts])


def xhc_stack_fwd(sh, X, outs, convs, Ws, idxs, workspace, x_ins=None, saveds=None, stream=None):
    """Forward of a stack of L = len(outs) sublayers on X in place, each
    sublayer's update fused with the next one's coefficient projection (see
    the C header).  ``convs``: None, or a list of L (w4, w8, w12) tuples or
    Nones (all sublayers with conv weights, or none); ``idxs``: L index
    lists; ``x_ins`` / ``saveds``: None or lists of L tensors (or Nones)."""
    L = len(outs)
    flat = [int(a) for ix in idxs for a in ix]
    if convs is None or all(c is None for c in convs):
        w4 = w8 = w12 = None
    else:
        w4, w8, w12 = (_ptr_array([None if c is None else c[j] for c in convs]) for j in range(3))
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("xhc_stack_fwd", LIB.xhc_stack_fwd(ctypes.byref(sh), L, _p(X), _ptr_array(outs), w4, w8, w12,
                                              _ptr_array(Ws), _idx(flat), _ptr_array(x_ins), _ptr_array(saveds),
                                              _p(workspace), ws_bytes, _s(stream)))


def xhc_fwd_routed_workspace_bytes(sh) -> int:
    return LIB.xhc_fwd_routed_workspace_bytes(ctypes.byref(sh))


def xhc_sublayer_fwd_routed(sh, X_in, X_out, out, conv, W, W_r, fixed, tok_idx, rrec, workspace, x_in=None,
                            saved=None, saved_active=None, stream=None):
    """The update with per-token active sets from the router (see the C
    header): ``fixed`` is the host list of always-active streams; ``tok_idx``
    [B,S,k] int32 and the router record ``rrec`` [B,S,2N+2] fp32 (scores,
    logits, LayerNorm mean and sd) are written."""
    w4, w8, w12 = _conv(conv)
    fixed = [int(a) for a in fixed]
    fx = (ctypes.c_int32 * max(len(fixed), 1))(*fixed) if fixed else None
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("xhc_sublayer_fwd_routed",
           LIB.xhc_sublayer_fwd_routed(ctypes.byref(sh), _p(X_in), _p(X_out), _p(out), w4, w8, w12, _p(W),
                                       _p(W_r), fx, len(fixed), _p(x_in), _p(saved), _p(saved_active),
                                       _p(tok_idx), _p(rrec), _p(workspace), ws_bytes, _s(stream)))


def xhc_bwd_routed_workspace_bytes(sh) -> int:
    return LIB.xhc_bwd_routed_workspace_bytes(ctypes.byref(sh))


def xhc_sublayer_bwd_routed(sh, X_state, out, conv, W, W_r, fixed, saved, tok_idx, rrec, dXp, dx_in, dX, dout, dconv,
                            dW, dW_r, workspace, saved_active=None, stream=None):
    """Reverse of xhc_sublayer_fwd_routed (see the C header).  Without
    ``saved_active`` X_state is the state before the update; with it, the
    state after an in-place forward, which the call turns back into the state
    before the update."""
    w4, w8, w12 = _conv(conv)
    d4, d8, d12 = _conv(dconv)
    fixed = [int(a) for a in fixed]
    fx = (ctypes.c_int32 * max(len(fixed), 1))(*fixed) if fixed else None
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("xhc_sublayer_bwd_routed",
           LIB.xhc_sublayer_bwd_routed(ctypes.byref(sh), _p(X_state), _p(saved_active), _p(out), w4, w8, w12, _p(W), _p(W_r), fx,
                                       len(fixed), _p(saved), _p(tok_idx), _p(rrec), _p(dXp), _p(dx_in), _p(dX),
                                       _p(dout), d4, d8, d12, _p(dW), _p(dW_r), _p(workspace), ws_bytes,
                                       _s(stream)))


def xhc_hres_active_weights(sh, W_pp, W_ra, idx, W, stream=None):
    """Full projection W [P, N*C] for H^res logits from the k active rows
    only: W_pp [N+4k, N*C] and W_ra [k*k, k*C] (see the C header)."""
    _check("xhc_hres_active_weights",
           LIB.xhc_hres_active_weights(ctypes.byref(sh), _p(W_pp), _p(W_ra), _idx(idx), _p(W), _s(stream)))


def xhc_hres_active_grad(sh, dW, idx, dW_ra, stream=None):
    """dL/dW_ra [k*k, k*C] from the full projection's gradient dW."""
    _check("xhc_hres_active_grad", LIB.xhc_hres_active_grad(ctypes.byref(sh), _p(dW), _idx(idx), _p(dW_ra),
                                                            _s(stream)))


def xhc_copy(src: Tensor, dst: Tensor, nbytes: Optional[int] = None, stream=None):
    n = src.numel() * src.element_size() if nbytes is None else nbytes
    _check("xhc_copy", LIB.xhc_copy(_p(src), _p(dst), n, _s(stream)))


def workspace(nbytes: int, device="cuda") -> Tensor:
    """A caller-owned workspace buffer (uint8) of at least ``nbytes`` bytes."""
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def xhc_timing_enable(on: bool = True):
    LIB.xhc_timing_enable(1 if on else 0)


def xhc_timing_collect(max_kernels: int = 64) -> dict:
    """{kernel name: (launches, total ms)} since the last collect."""
    names = ctypes.create_string_buffer(48 * max_kernels)
    counts = (ctypes.c_int * max_kernels)()
    ms = (ctypes.c_float * max_kernels)()
    n = LIB.xhc_timing_collect(names, counts, ms, max_kernels)
    if n < 0:
        raise XhcError("xhc_timing_collect", -n, LIB)
    raw = names.raw
    out = {}
    for i in range(n):
        nm = raw[48 * i: 48 * i + 48].split(b"\0", 1)[0].decode()
        out[nm] = (int(counts[i]), float(ms[i]))
    return out
