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
import pytest

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


@pytest.mark.parametrize("N,k,fixed", [(8, 3, [4, 1]), (6, 4, [2]), (16, 4, [])])
def test_score_scales_the_routed_write_back(N, k, fixed):
    """Closed form of the routed update.  With W = 0 every coefficient is
    fixed: H^pre = H^post = 1/2 and H^res = J/k.  With the K = 4 branch a delta
    at tap 1 and the other branches zero, the components are u_0 = out[t],
    u_1 = out[t - 1] (zero at t = 0), u_2 = u_3 = 0.  A one-hot W_r makes each
    router logit a chosen entry of the LayerNorm-ed state, written out here
    from its definition.  So every active slot gets the mean of the active
    rows, plus the write-back (out[t] + out[t - 1]) / 2, times the stream's
    score for a routed slot and times 1 for a fixed slot."""
    S, C, eps = 7, 5, 1e-6
    rng = np.random.default_rng(150 + N)
    X = rng.standard_normal((1, S, N, C))
    out = rng.standard_normal((1, S, C))
    W = np.zeros((xo.n_logits(N, k), N * C))
    conv = (np.zeros((C, 4)), np.zeros((C, 8)), np.zeros((C, 12)))
    conv[0][:, 1] = 1.0
    cols = rng.permutation(N * C)[:N]
    W_r = np.zeros((N, N * C))
    W_r[np.arange(N), cols] = 3.0
    r = xo.forward_routed(X, out, conv, W, W_r, fixed, k, eps=eps)
    want = X[0].copy()
    for t in range(S):
        v = X[0, t].reshape(-1)
        y = (v - v.mean()) / np.sqrt(((v - v.mean()) ** 2).mean() + eps)
        logit = 3.0 * y[cols]
        score = 1.0 / (1.0 + np.exp(-logit))
        others = [n for n in range(N) if n not in fixed]
        routed = sorted(others, key=lambda n: -logit[n])[: k - len(fixed)]
        active = list(fixed) + routed
        assert list(r["idx"][0, t]) == active
        mean = X[0, t, active].mean(axis=0)
        wb = 0.5 * (out[0, t] + (out[0, t - 1] if t > 0 else 0.0))
        for a in fixed:
            want[t, a] = mean + wb
        for a in routed:
            want[t, a] = mean + score[a] * wb
    np.testing.assert_allclose(r["Xp"][0], want, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r["x_in"][0], 0.5 * X[0].sum(axis=1), rtol=1e-12, atol=1e-12)


def test_given_active_sets_are_used():
    """An explicit active-set override reproduces the routed update for that
    set: with the router's own choice it equals the default, and with the
    routed slots swapped (a different but well-formed set) the rows move with
    the slots."""
    X, out, cv, W, _ = case(B=1, S=6, N=8, C=3, k=4, seed=151)
    W_r = _router(8, 3, 152)
    fixed = [3, 6]
    r = xo.forward_routed(X, out, cv, W, W_r, fixed, 4)
    r2 = xo.forward_routed(X, out, cv, W, W_r, fixed, 4, idx=r["idx"])
    np.testing.assert_array_equal(r["Xp"], r2["Xp"])
    swapped = r["idx"].copy()
    swapped[..., [2, 3]] = swapped[..., [3, 2]]
    r3 = xo.forward_routed(X, out, cv, W, W_r, fixed, 4, idx=swapped)
    assert (r3["idx"] == swapped).all()
    assert not np.allclose(r3["Xp"], r["Xp"])


def test_selection_check_accepts_valid_and_rejects_wrong_choices():
    """The GPU tests' validity check of router selections: the oracle's own
    choice passes; a wrong fixed slot, a repeated stream, routed slots out of
    order and an outranked choice each fail; a swap at an exact tie passes."""
    from tests.xhc_testlib import check_selection
    rng = np.random.default_rng(153)
    B, S, N, k, fixed = 2, 9, 8, 4, [5, 1]
    r = rng.standard_normal((B, S, N))
    s = 1.0 / (1.0 + np.exp(-r))
    own = np.stack([xo.route(s[b], fixed, k) for b in range(B)])
    assert check_selection(own, r, fixed, k, 1e-9) == 1.0
    bad = []
    g = own.copy(); g[0, 3, 0] = (g[0, 3, 0] + 1) % N; bad.append(g)          # fixed slot changed
    g = own.copy(); g[1, 2, 3] = g[1, 2, 2]; bad.append(g)                    # repeated stream
    g = own.copy(); g[0, 0, [2, 3]] = g[0, 0, [3, 2]]; bad.append(g)          # routed slots out of order
    g = own.copy()
    rest = [n for n in range(N) if n not in g[1, 4]]
    g[1, 4, 2] = min(rest, key=lambda n: r[1, 4, n]); bad.append(g)           # the weakest stream chosen
    for g in bad:
        with pytest.raises(AssertionError):
            check_selection(g, r, fixed, k, 1e-9)
    # an exact tie between the two routed slots: either order is valid
    r2 = r.copy()
    a, b_ = own[0, 6, 2], own[0, 6, 3]
    r2[0, 6, b_] = r2[0, 6, a]
    g = own.copy(); g[0, 6, [2, 3]] = g[0, 6, [3, 2]]
    check_selection(g, r2, fixed, k, 1e-9)
    check_selection(own, r2, fixed, k, 1e-9)
