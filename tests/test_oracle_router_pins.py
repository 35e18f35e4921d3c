"""Pins of the oracle's router with per-token active sets.

Source: "xHC: Expanded Hyper-Connections" (qingkeai.online), section "Dense
read, sparse write": the router reads the LayerNorm-ed whole state and gives
each stream a sigmoid score; fixed streams are always active, the others are
chosen per token by top-k; a routed stream's score multiplies its new
write-back; unchosen scores get no gradient.

Each test checks the oracle against something other than itself: the plain
update when every slot is fixed, the top-k property of the selection, the
LayerNorm statistics, and central finite differences of the backward.
"""
import numpy as np

from oracle import xhc_oracle as xo
from tests.test_oracle_pins import case, fd


def _router(N, C, seed, std=0.3):
    return np.random.default_rng(seed).standard_normal((N, N * C)) * std


def test_all_fixed_is_the_plain_update():
    X, out, cv, W, idx = case(B=2, S=9, N=16, C=4, k=4, seed=140, wstd=0.2)
    W_r = _router(16, 4, 141)
    r = xo.forward_routed(X, out, cv, W, W_r, list(idx), 4)
    p = xo.forward(X, out, cv, W, idx)
    np.testing.assert_array_equal(r["Xp"], p["Xp"])
    assert (r["idx"] == np.asarray(idx)[None, None, :]).all()
    dXp = np.random.default_rng(142).standard_normal(X.shape)
    gr = xo.backward_routed(X, out, cv, W, W_r, list(idx), 4, dXp)
    gp = xo.backward(X, out, cv, W, idx, dXp)
    for key in ("dX", "dout", "dW"):
        np.testing.assert_allclose(gr[key], gp[key], rtol=1e-13, atol=1e-13)
    assert not gr["dW_r"].any()


def test_selection_is_fixed_then_top_scores():
    X, out, cv, W, _ = case(B=1, S=20, N=16, C=3, k=4, seed=143)
    W_r = _router(16, 3, 144)
    fixed = [5, 2]
    r = xo.forward_routed(X, out, cv, W, W_r, fixed, 4)
    s, idx = r["s"][0], r["idx"][0]
    for t in range(idx.shape[0]):
        assert list(idx[t, :2]) == fixed
        routed = list(idx[t, 2:])
        rest = [n for n in range(16) if n not in fixed and n not in routed]
        assert s[t, routed[0]] >= s[t, routed[1]]
        assert min(s[t, routed]) >= max(s[t, rest])
    # the unchosen streams are left as they were
    inactive = np.ones((20, 16), dtype=bool)
    np.put_along_axis(inactive, idx, False, axis=1)
    np.testing.assert_array_equal(r["Xp"][0][inactive], X[0][inactive])


def test_layernorm_statistics():
    X, *_ = case(B=1, S=7, N=16, C=5, k=4, seed=145)
    W_r = np.zeros((16, 80))
    cols = np.random.default_rng(146).permutation(80)[:16]
    W_r[np.arange(16), cols] = 1.0                    # r_n = y[col_n]
    s, r, y, sd = xo.router_scores(X[0], W_r, 1e-6)
    np.testing.assert_allclose(y.mean(axis=1), 0.0, atol=1e-13)
    var = X[0].reshape(7, -1).var(axis=1)
    np.testing.assert_allclose((y * y).mean(axis=1), var / (var + 1e-6), rtol=1e-12)
    np.testing.assert_array_equal(r, y[:, cols])
    np.testing.assert_allclose(s, 1.0 / (1.0 + np.exp(-r)), rtol=1e-15)


def test_routed_backward_finite_differences():
    B, S, N, C, k = 1, 12, 16, 3, 4
    X, out, cv, W, _ = case(B=B, S=S, N=N, C=C, k=k, seed=147, wstd=0.3, cstd=0.4)
    W_r = _router(N, C, 148)
    fixed = [0, 9]
    rng = np.random.default_rng(149)
    dXp = rng.standard_normal(X.shape)
    dxi = rng.standard_normal(out.shape)
    g = xo.backward_routed(X, out, cv, W, W_r, fixed, k, dXp, dxi)
    base = xo.forward_routed(X, out, cv, W, W_r, fixed, k)["idx"]

    def L():
        r = xo.forward_routed(X, out, cv, W, W_r, fixed, k)
        # the active sets are piecewise constant: a step must not move them
        assert (r["idx"] == base).all()
        return (r["Xp"] * dXp).sum() + (r["x_in"] * dxi).sum()

    num, _ = fd(L, out)
    np.testing.assert_allclose(g["dout"], num, rtol=1e-6, atol=1e-7)
    for w, dw in zip(cv, g["dconv"]):
        num, _ = fd(L, w)
        np.testing.assert_allclose(dw, num, rtol=1e-6, atol=1e-7)
    for A, key in ((X, "dX"), (W, "dW"), (W_r, "dW_r")):
        picks = [tuple(rng.integers(0, n) for n in A.shape) for _ in range(30)]
        num, it = fd(L, A, picks=picks)
        for ix in it:
            assert abs(num[ix] - g[key][ix]) <= 1e-6 * max(1.0, abs(num[ix])), (key, ix)
