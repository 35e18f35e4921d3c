"""The C-ABI library loads, exports every symbol include/xhc.h declares, and
rejects bad arguments on the host before any launch (no GPU needed: every
call below returns from host-side validation)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "xhc.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(xhc_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from residual_stream_expansion_xhc_b300 import _lib
    return _lib


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib.LIB, n), n
    assert set(names) == set(lib.EXPORTS)
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True, text=True).stdout
    for n in names:
        assert re.search(rf"\bT {n}$", out, flags=re.M), n


def shape(lib, B=2, S=8, N=16, C=256, k=4, dtype=1, iters=20, eps=1e-6):
    return lib.XhcShape(B, S, N, C, k, dtype, iters, eps)


FAKE = ctypes.c_void_p(1 << 20)        # 16-byte aligned, never dereferenced on the host
MIS = ctypes.c_void_p((1 << 20) + 8)   # misaligned


def idx(*v):
    return (ctypes.c_int32 * len(v))(*v)


def fwd(lib, sh, ix, X=FAKE, W=FAKE, conv=(None, None, None), ws=None, ws_bytes=0, saved=None):
    return lib.LIB.xhc_sublayer_fwd(ctypes.byref(sh), X, X, FAKE, conv[0], conv[1], conv[2], W, ix, None, saved,
                                    None, ws, ws_bytes, None)


def test_status_strings(lib):
    for s in range(9):
        assert lib.LIB.xhc_status_string(s)
    assert lib.LIB.xhc_status_string(99) == b"unknown status"


def test_num_logits(lib):
    assert lib.LIB.xhc_num_logits(ctypes.byref(shape(lib))) == 48
    assert lib.LIB.xhc_num_logits(ctypes.byref(shape(lib, N=4, k=4))) == 36


@pytest.mark.parametrize("kw,status", [
    (dict(N=17), 1), (dict(N=0), 1), (dict(k=5), 1), (dict(k=0), 1), (dict(N=3, k=4), 1),
    (dict(iters=65), 1), (dict(iters=-1), 1), (dict(eps=0.0), 1), (dict(B=-1), 1),
    (dict(dtype=7), 4), (dict(C=100), 3), (dict(C=6, dtype=0), 3)])
def test_shape_rejected(lib, kw, status):
    sh = shape(lib, **kw)
    assert fwd(lib, sh, idx(0, 1, 2, 3)) == status


@pytest.mark.parametrize("ix", [(0, 1, 2, 2), (0, 1, 2, 16), (-1, 1, 2, 3)])
def test_index_rejected(lib, ix):
    assert fwd(lib, shape(lib), idx(*ix)) == 2


def test_null_and_alignment_rejected(lib):
    sh = shape(lib)
    assert fwd(lib, sh, idx(0, 1, 2, 3), X=None) == 8
    assert fwd(lib, sh, idx(0, 1, 2, 3), X=MIS) == 3
    assert fwd(lib, sh, None) == 2
    # conv weights: all three or none
    assert fwd(lib, sh, idx(0, 1, 2, 3), conv=(FAKE, None, FAKE)) == 8
    # no saved coefficients and no workspace
    assert fwd(lib, sh, idx(0, 1, 2, 3)) == 5
    need = lib.LIB.xhc_fwd_workspace_bytes(ctypes.byref(sh))
    assert need >= 2 * 8 * 49 * 4
    assert fwd(lib, sh, idx(0, 1, 2, 3), ws=FAKE, ws_bytes=need - 1) == 5
    # with the logits kept by the caller, the bf16 path still needs the coefficient block
    assert fwd(lib, sh, idx(0, 1, 2, 3), saved=FAKE) == 5


def test_forward_workspace_sizes(lib):
    L = lib.LIB
    sh = shape(lib, B=3, S=100)                       # bf16, 300 tokens, P = 48, C = 256
    up = lambda b: (b + 255) // 256 * 256             # noqa: E731
    coef, z = up(300 * 48 * 4), up(300 * 49 * 4)
    wsplit = up(2 * 48 * 16 * 256 * 2)                # bf16 hi and lo parts of W, 48 rows each
    assert L.xhc_fwd_workspace_need(ctypes.byref(sh), 1) == coef + wsplit
    assert L.xhc_fwd_workspace_need(ctypes.byref(sh), 0) == coef + wsplit + z
    assert L.xhc_fwd_workspace_bytes(ctypes.byref(sh)) == coef + wsplit + z
    f32 = shape(lib, B=3, S=100, dtype=0)             # the fp32 path keeps no coefficient block
    assert L.xhc_fwd_workspace_need(ctypes.byref(f32), 1) == 0
    assert L.xhc_fwd_workspace_need(ctypes.byref(f32), 0) == z


def test_empty_forward_launches_nothing(lib):
    sh = shape(lib, B=0)
    assert fwd(lib, sh, idx(0, 1, 2, 3)) == 0


def test_backward_rejections(lib):
    sh = shape(lib)
    L = lib.LIB
    need = L.xhc_bwd_workspace_bytes(ctypes.byref(sh))
    assert need > 0
    args = dict(X=FAKE, act=None, out=FAKE, w=(None, None, None), W=FAKE, saved=FAKE, dXp=ctypes.c_void_p(1 << 22), dxi=None, dX=FAKE,
                dout=FAKE, dw=(None, None, None), dW=FAKE, ws=FAKE, wsb=need)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return L.xhc_sublayer_bwd(ctypes.byref(sh), a["X"], a["act"], a["out"], *a["w"], a["W"], idx(0, 1, 2, 3),
                                  a["saved"], a["dXp"], a["dxi"], a["dX"], a["dout"], *a["dw"], a["dW"], a["ws"],
                                  a["wsb"], None)
    assert call(wsb=need - 1) == 5
    assert call(ws=None) == 5
    assert call(w=(FAKE, FAKE, FAKE)) == 8               # conv weights without their gradients
    assert call(act=FAKE, saved=None) == 8               # recomputation needs the pre-update state
    assert call(dW=MIS) == 3
    assert call(dX=ctypes.c_void_p(1 << 21), dXp=ctypes.c_void_p(1 << 21)) == 8   # dX may not alias dX'


def test_copy_rejections(lib):
    assert lib.LIB.xhc_copy(FAKE, FAKE, 24, None) == 3
    assert lib.LIB.xhc_copy(None, FAKE, 32, None) == 8
    assert lib.LIB.xhc_copy(FAKE, FAKE, 0, None) == 0


# ---------------------------------------------------------------- Gram-Schmidt flag

def gs_shape(lib, **kw):
    sh = shape(lib, **kw)
    sh.gram_schmidt = 1
    return sh


def test_gram_schmidt_flag_validated(lib):
    sh = shape(lib)
    sh.gram_schmidt = 2
    assert fwd(lib, sh, idx(0, 1, 2, 3)) == 1
    assert lib.LIB.xhc_fwd_workspace_bytes(ctypes.byref(sh)) == 0


def test_gram_schmidt_workspace_sizes(lib):
    L = lib.LIB
    up = lambda b: (b + 255) // 256 * 256             # noqa: E731
    plain, gs = shape(lib, B=3, S=100, C=512), gs_shape(lib, B=3, S=100, C=512)
    gpart = up(300 * 2 * 12 * 4)                      # 12 floats per token and 256-channel block
    for keeps in (0, 1):
        assert L.xhc_fwd_workspace_need(ctypes.byref(gs), keeps) == L.xhc_fwd_workspace_need(ctypes.byref(plain), keeps) + gpart
    assert L.xhc_bwd_workspace_bytes(ctypes.byref(gs)) > L.xhc_bwd_workspace_bytes(ctypes.byref(plain)) + gpart


def test_gram_schmidt_rejections(lib):
    L = lib.LIB
    conv = (FAKE, FAKE, FAKE)
    # the fp32 path and a C the tensor-core passes do not tile have no Gram-Schmidt
    assert fwd(lib, gs_shape(lib, dtype=0), idx(0, 1, 2, 3), conv=conv) == 4
    assert fwd(lib, gs_shape(lib, C=72), idx(0, 1, 2, 3), conv=conv) == 4
    # without conv weights the flag changes nothing (missing workspace reported as usual)
    assert fwd(lib, gs_shape(lib, dtype=0), idx(0, 1, 2, 3)) == 5
    # building blocks handle raw components only
    sh = gs_shape(lib)
    assert L.xhc_tfa(ctypes.byref(sh), FAKE, FAKE, FAKE, FAKE, FAKE, None) == 8
    assert L.xhc_sparse_update(ctypes.byref(sh), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                               idx(0, 1, 2, 3), None) == 8


# ---------------------------------------------------------------- router entry points

def test_router_rejections(lib):
    L = lib.LIB
    sh = shape(lib)
    need = L.xhc_fwd_routed_workspace_bytes(ctypes.byref(sh))
    assert need > L.xhc_fwd_workspace_bytes(ctypes.byref(sh))

    def fwd_r(sh, fixed, nf, ws=FAKE, wsb=None):
        fx = (ctypes.c_int32 * 4)(*fixed) if fixed is not None else None
        return L.xhc_sublayer_fwd_routed(ctypes.byref(sh), FAKE, FAKE, FAKE, None, None, None, FAKE, FAKE, fx, nf,
                                         None, None, None, FAKE, FAKE, ws, need if wsb is None else wsb, None)
    assert fwd_r(sh, (0, 1, 0, 0), 2, wsb=need - 1) == 5
    assert fwd_r(sh, (0, 0, 0, 0), 2) == 2            # repeated fixed stream
    assert fwd_r(sh, (0, 16, 0, 0), 2) == 2           # outside [0, N)
    assert fwd_r(sh, (0, 1, 2, 3), 5) == 2            # more fixed streams than slots
    assert fwd_r(shape(lib, dtype=0), (0, 1, 0, 0), 2) == 4
    gs = shape(lib)
    gs.gram_schmidt = 1
    assert fwd_r(gs, (0, 1, 0, 0), 2) == 8
    bneed = L.xhc_bwd_routed_workspace_bytes(ctypes.byref(sh))
    assert bneed > L.xhc_bwd_workspace_bytes(ctypes.byref(sh))
    fx = (ctypes.c_int32 * 2)(0, 1)
    # P + N > 64 has no room for the router rows in the backward (N = 16, k = 4 fits; N = 8, k = 4 fits;
    # N = 12, k = 4: P = 44, 44 + 12 = 56 fits) -- fp32 is refused
    assert L.xhc_sublayer_bwd_routed(ctypes.byref(shape(lib, dtype=0)), FAKE, None, FAKE, None, None, None, FAKE,
                                     FAKE, fx, 2, FAKE, FAKE, FAKE, ctypes.c_void_p(1 << 22), None, FAKE, FAKE, None, None,
                                     None, FAKE, FAKE, FAKE, bneed, None) == 4


# ---------------------------------------------------------------- fused stack forward

def test_stack_rejections(lib):
    L = lib.LIB
    sh = shape(lib)
    need = L.xhc_stack_fwd_workspace_bytes(ctypes.byref(sh))
    # two coefficient blocks, the bf16 split of one W, the tap-major conv weights
    assert need >= 2 * 16 * 48 * 4 + 2 * 48 * 16 * 256 * 2 + 24 * 256 * 4

    def arr(n, v=FAKE):
        return (ctypes.c_void_p * n)(*([v.value] * n))

    def stack(sh, nl, ix, conv=True, wsb=None, outs=None, Ws=None, x=FAKE):
        c = (arr(nl), arr(nl), arr(nl)) if conv else (None, None, None)
        return L.xhc_stack_fwd(ctypes.byref(sh), nl, x, arr(nl) if outs is None else outs, *c,
                               arr(nl) if Ws is None else Ws, ix, None, None, FAKE,
                               need if wsb is None else wsb, None)
    good = idx(0, 1, 2, 3, 4, 5, 6, 7)
    assert stack(sh, 2, good, wsb=need - 1) == 5                         # workspace too small
    assert stack(sh, 0, good) == 8                                       # no sublayer
    assert stack(sh, 2, idx(0, 1, 2, 3, 4, 4, 6, 7)) == 2                # repeated stream in sublayer 1
    assert stack(sh, 2, idx(0, 1, 2, 3, 4, 5, 6, 16)) == 2               # outside [0, N)
    assert stack(shape(lib, dtype=0), 2, good) == 4                      # fp32 state
    assert stack(shape(lib, C=96), 2, good) == 1                         # C not a multiple of 64
    assert stack(sh, 2, good, x=MIS) == 3                                # misaligned state
    assert stack(sh, 2, good, outs=(ctypes.c_void_p * 2)(FAKE.value, None)) == 8   # missing out
    assert stack(sh, 2, good, Ws=(ctypes.c_void_p * 2)(FAKE.value, MIS.value)) == 3
    part = (ctypes.c_void_p * 2)(FAKE.value, None)
    assert L.xhc_stack_fwd(ctypes.byref(sh), 2, FAKE, arr(2), arr(2), arr(2), part, arr(2), good, None, None, FAKE,
                           need, None) == 8                               # sublayer 1: two of three conv weights
    assert L.xhc_stack_fwd(ctypes.byref(sh), 2, FAKE, arr(2), arr(2), None, None, arr(2), good, None, None, FAKE,
                           need, None) == 8                               # conv arrays: all three or none
    empty = shape(lib, B=0)
    assert stack(empty, 2, good, wsb=0) == 0                             # nothing to do


def test_debug_library_exports_the_same_symbols():
    """The bounds-checked build (libxhc_debug.so) loads on a machine without a
    GPU and exports every entry point the header declares."""
    import os
    from residual_stream_expansion_xhc_b300 import build
    if not os.path.exists(build.LIB_DEBUG):
        pytest.skip("debug build not built")
    names = declared_functions()
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB_DEBUG], capture_output=True, text=True).stdout
    for n in names:
        assert re.search(rf"\bT {n}$", out, flags=re.M), n
    ctypes.CDLL(build.LIB_DEBUG)
