"""Pins of the CPU oracle against facts fixed by the pages and by mathematics.

Sources: "xHC: Expanded Hyper-Connections" (qingkeai.online research
retrospective) sections "Scaling N" (state X in R^{N x C}, H^pre / H^post /
H^res, Sinkhorn), "Write-back bottleneck" (mHC write h^post_i * out),
"Temporal Feature Augmentation" (causal depthwise convs K = 4, 8, 12 stacked
with the raw output), "Dense read, sparse write" (only the k active streams
are written; inactive streams are unchanged).

None of these tests compares the oracle with a retyped copy of itself: each
checks a closed form, an exact hand-worked value, an invariant, a special case
or finite differences.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import xhc_oracle as xo

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


def case(B=2, S=16, N=16, C=8, k=4, seed=0, wstd=0.05, cstd=0.2, conv=True):
    X = rnd((B, S, N, C), seed)
    out = rnd((B, S, C), seed + 1)
    cv = tuple(rnd((C, K), seed + 2 + i, cstd) for i, K in enumerate(xo.CONV_KS)) if conv else None
    W = rnd((xo.n_logits(N, k), N * C), seed + 5, wstd)
    idx = np.random.default_rng(seed + 6).permutation(N)[:k]
    return X, out, cv, W, idx


# ---------------------------------------------------------------- Sinkhorn

def read_golden():
    rows = []
    with open(os.path.join(GOLDEN, "sinkhorn_worked.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            name, k, it, m0, h = [s.strip() for s in line.split("|")]
            k, it = int(k), int(it)
            m0 = np.array([float(x) for x in m0.split()]).reshape(k, k)
            h = np.array([float(Fraction(x)) for x in h.split()]).reshape(k, k)
            rows.append((name, it, m0, h))
    return rows


@pytest.mark.parametrize("name,iters,m0,h", read_golden())
def test_sinkhorn_hand_worked(name, iters, m0, h):
    # feed log(M0) as logits: exp(Z - max Z) is M0 up to a common factor,
    # which the first row normalisation removes exactly
    H, _ = xo.sinkhorn(np.log(m0), iters)
    np.testing.assert_allclose(H, h, rtol=0, atol=1e-14)


def test_sinkhorn_columns_exact_rows_converge():
    Z = rnd((2000, 4, 4), 3, 3.6)
    H, _ = xo.sinkhorn(Z, 20)
    assert np.abs(H.sum(axis=-2) - 1).max() < 1e-12       # last step: columns
    Zs = rnd((2000, 4, 4), 4, 0.5)                         # converged regime
    Hs, _ = xo.sinkhorn(Zs, 20)
    assert np.abs(Hs.sum(axis=-1) - 1).max() < 1e-6
    assert np.abs(Hs.sum(axis=-2) - 1).max() < 1e-12
    assert (H > 0).all()


def test_sinkhorn_additive_logits_uniform():
    a = rnd((50, 4, 1), 5)
    b = rnd((50, 1, 4), 6)
    H, _ = xo.sinkhorn(a + b, 1)
    np.testing.assert_allclose(H, np.full((50, 4, 4), 0.25), atol=1e-14)


def test_sinkhorn_reverse_finite_differences():
    Z = rnd((3, 4, 4), 7, 1.5)
    dH = rnd((3, 4, 4), 8)
    H, tr = xo.sinkhorn(Z, 20)
    dZ = xo.sinkhorn_reverse(dH, tr)
    h = 1e-6
    num = np.zeros_like(Z)
    for idx in np.ndindex(*Z.shape):
        Zp = Z.copy(); Zp[idx] += h
        Zm = Z.copy(); Zm[idx] -= h
        num[idx] = ((xo.sinkhorn(Zp, 20)[0] - xo.sinkhorn(Zm, 20)[0]) * dH).sum() / (2 * h)
    np.testing.assert_allclose(dZ, num, rtol=1e-6, atol=1e-9)
    # a shift of one row of logits is removed by the row normalisation
    assert np.abs(dZ.sum(axis=-1)).max() < 1e-12


# ---------------------------------------------------------------- forward closed forms

def test_zero_projection_closed_form():
    X, out, cv, W, idx = case(seed=10)
    W = np.zeros_like(W)
    r = xo.forward(X, out, cv, W, idx)
    k = len(idx)
    assert np.all(r["hpre"] == 0.5) and np.all(r["hpost"] == 0.5)
    np.testing.assert_allclose(r["hres"], 1.0 / k, atol=1e-15)
    np.testing.assert_allclose(r["x_in"], 0.5 * X.sum(axis=2), atol=1e-12)
    u = r["u"]                                          # [B, 4, S, C]
    expect = X[:, :, idx, :].mean(axis=2) + 0.5 * u.sum(axis=1)
    for i, a in enumerate(idx):
        np.testing.assert_allclose(r["Xp"][:, :, a, :], expect, atol=1e-12)


def test_rmsnorm_scale_closed_form():
    # every entry of the state equal to a: mean(v^2) = a^2 over all N*C
    B, S, N, C, k = 1, 3, 4, 8, 2
    a = 0.37
    X = np.full((B, S, N, C), a)
    out = np.zeros((B, S, C))
    W = np.zeros((xo.n_logits(N, k), N * C))
    q, m = 5, 17                          # one logit reading one state entry
    W[q, m] = 1.0
    r = xo.forward(X, out, None, W, [0, 1])
    z = r["z"][0]
    np.testing.assert_allclose(z[:, q], a / np.sqrt(a * a + 1e-6), rtol=1e-15)
    assert np.count_nonzero(z) == S
    np.testing.assert_allclose(r["rstd"], 1.0 / np.sqrt(a * a + 1e-6), rtol=1e-15)


def test_logit_layout():
    # row N + 4i + c drives H^post[i, c]; row N + 4k + k i + j drives Z[i, j]
    B, S, N, C, k = 1, 1, 4, 4, 2
    X = np.zeros((B, S, N, C)); X[0, 0, 1, 2] = 1.0          # v[1*C + 2] = 1
    out = np.ones((B, S, C))
    P = xo.n_logits(N, k)
    col = 1 * C + 2
    W = np.zeros((P, N * C))
    W[2, col] = 4.0                      # H^pre[2]
    W[N + 4 * 1 + 3, col] = 5.0          # H^post[1, 3]
    W[N + 4 * k + k * 1 + 0, col] = 6.0  # H^res logit [1, 0]
    r = xo.forward(X, out, None, W, [0, 3])
    rs = r["rstd"][0, 0]
    hp = np.full(N, 0.5); hp[2] = xo.sigmoid(4.0 * rs)
    np.testing.assert_allclose(r["hpre"][0, 0], hp, rtol=1e-15)
    hq = np.full((k, 4), 0.5); hq[1, 3] = xo.sigmoid(5.0 * rs)
    np.testing.assert_allclose(r["hpost"][0, 0], hq, rtol=1e-15)
    Z = np.zeros((k, k)); Z[1, 0] = 6.0 * rs
    np.testing.assert_allclose(r["z"][0, 0, N + 4 * k:].reshape(k, k), Z, rtol=1e-15)


def test_mix_orientation_rows_are_output_slots():
    # X[a_j] = e_j (unit vectors over channels): X'[a_i][j] = H^res[i, j]
    B, S, N, C, k = 1, 1, 6, 4, 3
    X = np.zeros((B, S, N, C))
    idx = [4, 1, 2]
    for j, a in enumerate(idx):
        X[0, 0, a, j] = 1.0
    W = rnd((xo.n_logits(N, k), N * C), 3, 2.0)
    r = xo.forward(X, np.zeros((B, S, C)), None, W, idx, iters=3)
    H = r["hres"][0, 0]
    assert np.abs(H - H.T).max() > 1e-3          # a non-symmetric case
    for i, a in enumerate(idx):
        np.testing.assert_allclose(r["Xp"][0, 0, a, :k], H[i], rtol=0, atol=1e-15)


def test_delta_conv_shifts():
    B, S, N, C, k = 2, 20, 4, 5, 2
    X, out, cv, W, idx = case(B=B, S=S, N=N, C=C, k=k, seed=20)
    for j, K in enumerate(xo.CONV_KS):
        for tau in (0, K - 1):
            conv = [np.zeros((C, KK)) for KK in xo.CONV_KS]
            conv[j][:, tau] = 1.0
            u = xo.forward(X, out, tuple(conv), W, idx)["u"]
            expect = np.zeros((B, S, C))
            expect[:, tau:, :] = out[:, : S - tau, :]
            np.testing.assert_array_equal(u[:, j + 1], expect)
            for jj in range(1, 4):
                if jj != j + 1:
                    assert not u[:, jj].any()
            np.testing.assert_array_equal(u[:, 0], out)


def test_mhc_special_case():
    # zero conv branches, k = N, identity indices: X' = H^res X + h^post[:, 0] out^T
    B, S, N, C = 2, 9, 4, 6
    X, out, _, W, _ = case(B=B, S=S, N=N, C=C, k=N, seed=30, wstd=0.3)
    zero = tuple(np.zeros((C, K)) for K in xo.CONV_KS)
    idx = list(range(N))
    r = xo.forward(X, out, zero, W, idx)
    r2 = xo.forward(X, out, None, W, idx)
    for b in range(B):
        for t in range(S):
            H = r["hres"][b, t]
            hp = r["hpost"][b, t][:, 0]
            expect = H @ X[b, t] + np.outer(hp, out[b, t])
            np.testing.assert_allclose(r["Xp"][b, t], expect, rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(r["Xp"], r2["Xp"])


def test_inactive_rows_bit_identical():
    X, out, cv, W, idx = case(seed=40)
    r = xo.forward(X, out, cv, W, idx)
    inactive = [n for n in range(X.shape[2]) if n not in set(idx.tolist())]
    assert np.array_equal(r["Xp"][:, :, inactive], X[:, :, inactive])
    assert not np.array_equal(r["Xp"][:, :, idx], X[:, :, idx])


def test_causality_and_locality():
    B, S = 2, 30
    X, out, cv, W, idx = case(B=B, S=S, seed=50)
    base = xo.forward(X, out, cv, W, idx)["Xp"]
    t0 = 7
    out2 = out.copy(); out2[1, t0] += 1.0
    d = np.abs(xo.forward(X, out2, cv, W, idx)["Xp"] - base).sum(axis=(2, 3))
    assert not d[0].any()                            # other sequence untouched
    assert not d[1, :t0].any()                       # the past is untouched
    assert (d[1, t0:t0 + 12] > 0).all()              # K = 12 reaches 11 tokens ahead
    assert not d[1, t0 + 12:].any()
    X2 = X.copy(); X2[0, t0] += 0.5
    d = np.abs(xo.forward(X2, out, cv, W, idx)["Xp"] - base).sum(axis=(2, 3))
    assert d[0, t0] > 0 and np.count_nonzero(d) == 1


def test_batch_independence():
    X, out, cv, W, idx = case(B=3, seed=60)
    full = xo.forward(X, out, cv, W, idx)
    for b in range(3):
        one = xo.forward(X[b:b + 1], out[b:b + 1], cv, W, idx)
        np.testing.assert_array_equal(one["Xp"][0], full["Xp"][b])
        np.testing.assert_array_equal(one["x_in"][0], full["x_in"][b])


def test_index_equivariance():
    B, S, N, C, k = 1, 12, 8, 4, 4
    X, out, cv, W, idx = case(B=B, S=S, N=N, C=C, k=k, seed=70, wstd=0.3)
    perm = np.array([2, 0, 3, 1])
    idx2 = idx[perm]
    W2 = W.copy()
    for i2, i in enumerate(perm):
        W2[N + 4 * i2: N + 4 * i2 + 4] = W[N + 4 * i: N + 4 * i + 4]
        for j2, j in enumerate(perm):
            W2[N + 4 * k + k * i2 + j2] = W[N + 4 * k + k * i + j]
    a = xo.forward(X, out, cv, W, idx)["Xp"]
    b = xo.forward(X, out, cv, W2, idx2)["Xp"]
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-13)


def brute_force(X, out, conv, W, idx, iters=20, eps=1e-6):
    """Independent dense restatement for S <= 8: per channel the convolutions
    are S x S lower-banded Toeplitz matrices; per token the write is a dense
    N x N matrix (identity on inactive rows, H^res scattered to (a_i, a_j))
    plus an N x 4 matrix of H^post rows."""
    B, S, N, C = X.shape
    k = len(idx)
    Xp = np.zeros_like(X)
    for b in range(B):
        U = np.zeros((S, 4, C))
        for c in range(C):
            U[:, 0, c] = out[b, :, c]
            for j, w in enumerate(conv):
                T = np.zeros((S, S))
                for t in range(S):
                    for s in range(S):
                        if 0 <= t - s < w.shape[1]:
                            T[t, s] = w[c, t - s]
                U[:, j + 1, c] = T @ out[b, :, c]
        for t in range(S):
            v = X[b, t].reshape(-1)
            z = W @ v / np.sqrt(np.dot(v, v) / (N * C) + eps)
            hpost = 1 / (1 + np.exp(-z[N:N + 4 * k])).reshape(k, 4)
            M = np.exp(z[N + 4 * k:].reshape(k, k))
            for _ in range(iters):
                M = M / M.sum(axis=1, keepdims=True)
                M = M / M.sum(axis=0, keepdims=True)
            D = np.eye(N)
            Post = np.zeros((N, 4))
            for i, a in enumerate(idx):
                D[a, :] = 0.0
                for j, aj in enumerate(idx):
                    D[a, aj] = M[i, j]
                Post[a] = hpost[i]
            Xp[b, t] = D @ X[b, t] + Post @ U[t]
    return Xp


@pytest.mark.parametrize("S,N,k", [(1, 16, 4), (5, 16, 4), (8, 4, 4), (7, 6, 2)])
def test_brute_force_small(S, N, k):
    X, out, cv, W, idx = case(B=2, S=S, N=N, C=5, k=k, seed=80 + S, wstd=0.3)
    got = xo.forward(X, out, cv, W, idx)["Xp"]
    np.testing.assert_allclose(got, brute_force(X, out, cv, W, idx), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- backward

def loss(X, out, cv, W, idx, dXp, dx_in):
    r = xo.forward(X, out, cv, W, idx)
    val = (r["Xp"] * dXp).sum()
    if dx_in is not None:
        val += (r["x_in"] * dx_in).sum()
    return val


def fd(fn, A, h=1e-6, picks=None):
    g = np.zeros_like(A)
    it = picks if picks is not None else list(np.ndindex(*A.shape))
    for ix in it:
        old = A[ix]
        A[ix] = old + h; fp = fn()
        A[ix] = old - h; fm = fn()
        A[ix] = old
        g[ix] = (fp - fm) / (2 * h)
    return g, it


@pytest.mark.parametrize("N,k,with_dxin,conv", [(16, 4, True, True), (4, 4, False, True), (16, 4, False, False)])
def test_backward_finite_differences(N, k, with_dxin, conv):
    B, S, C = 1, 14, 3
    X, out, cv, W, idx = case(B=B, S=S, N=N, C=C, k=k, seed=90 + N, wstd=0.3, conv=conv)
    rng = np.random.default_rng(5)
    dXp = rng.standard_normal(X.shape)
    dxi = rng.standard_normal(out.shape) if with_dxin else None
    g = xo.backward(X, out, cv, W, idx, dXp, dxi)
    L = lambda: loss(X, out, cv, W, idx, dXp, dxi)
    picks = [tuple(rng.integers(0, s) for s in X.shape) for _ in range(40)]
    num, it = fd(L, X, picks=picks)
    for ix in it:
        assert abs(num[ix] - g["dX"][ix]) <= 1e-6 * max(1.0, abs(num[ix])), ix
    num, it = fd(L, out)
    np.testing.assert_allclose(g["dout"], num, rtol=1e-6, atol=1e-7)
    if conv:
        for w, dw in zip(cv, g["dconv"]):
            num, _ = fd(L, w)
            np.testing.assert_allclose(dw, num, rtol=1e-6, atol=1e-7)
    picks = [tuple(rng.integers(0, s) for s in W.shape) for _ in range(40)]
    num, it = fd(L, W, picks=picks)
    for ix in it:
        assert abs(num[ix] - g["dW"][ix]) <= 1e-6 * max(1.0, abs(num[ix])), ix


def test_backward_structure():
    X, out, cv, W, idx = case(seed=100, wstd=0.3)
    N, k = X.shape[2], len(idx)
    rng = np.random.default_rng(1)
    dXp = rng.standard_normal(X.shape)
    g = xo.backward(X, out, cv, W, idx, dXp, None, keep=True)
    dzres = g["dz"][..., N + 4 * k:].reshape(X.shape[0], X.shape[1], k, k)
    assert np.abs(dzres.sum(axis=-1)).max() < 1e-12           # row-shift invariance
    assert not g["dz"][..., :N].any()                          # no dx_in: H^pre gets no gradient
    # W = 0 and no dx_in: inactive rows of dX equal dX' bit for bit
    g0 = xo.backward(X, out, cv, np.zeros_like(W), idx, dXp, None)
    inactive = [n for n in range(N) if n not in set(idx.tolist())]
    assert np.array_equal(g0["dX"][:, :, inactive], dXp[:, :, inactive])
    # zero conv branches: dout = sum_i hpost[i, 0] G_i
    zero = tuple(np.zeros_like(w) for w in cv)
    gz = xo.backward(X, out, zero, W, idx, dXp, None)
    hpost = xo.forward(X, out, zero, W, idx)["hpost"]
    expect = np.einsum("bsi,bsic->bsc", hpost[..., 0], dXp[:, :, idx])
    np.testing.assert_allclose(gz["dout"], expect, rtol=1e-13, atol=1e-13)


def test_max_rel_err_definition():
    ref = np.array([1.0, -2.0, 1e-9, 0.0])
    rms = np.sqrt((1 + 4 + 1e-18) / 4)
    got = ref + np.array([0.01, 0.0, 0.001, 0.0])
    assert abs(xo.max_rel_err(got, ref) - max(0.01 / max(1.0, rms), 0.001 / rms)) < 1e-15


# ---------------------------------------------------------------- H^res from the active rows only

def test_hres_active_logits_definition():
    # z_res = rstd * vec(X[a_0], .., X[a_{k-1}]) . W_ra^T, the other logits over the whole state
    B, S, N, C, k = 1, 6, 16, 5, 4
    X, out, cv, _, idx = case(B=B, S=S, N=N, C=C, k=k, seed=130)
    rng = np.random.default_rng(3)
    W_pp = rng.standard_normal((N + 4 * k, N * C)) * 0.05
    W_ra = rng.standard_normal((k * k, k * C)) * 0.05
    r = xo.forward(X, out, cv, xo.expand_hres_active(W_pp, W_ra, idx, N, C), idx)
    v = X[0].reshape(S, N * C)
    va = X[0][:, list(idx), :].reshape(S, k * C)
    rstd = 1.0 / np.sqrt((v * v).mean(axis=1) + 1e-6)
    np.testing.assert_allclose(r["z"][0, :, : N + 4 * k], rstd[:, None] * (v @ W_pp.T), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r["z"][0, :, N + 4 * k:], rstd[:, None] * (va @ W_ra.T), rtol=1e-12, atol=1e-14)
    # the inactive streams' state does not reach the mixing logits
    X2 = X.copy()
    inactive = [n for n in range(N) if n not in idx]
    X2[:, :, inactive] *= 3.0
    r2 = xo.forward(X2, out, cv, xo.expand_hres_active(W_pp, W_ra, idx, N, C), idx)
    np.testing.assert_allclose(r2["z"][..., N + 4 * k:] / r2["rstd"][..., None],
                               r["z"][..., N + 4 * k:] / r["rstd"][..., None], rtol=1e-12)


def test_hres_active_gradient_finite_differences():
    B, S, N, C, k = 1, 8, 16, 3, 4
    X, out, cv, _, idx = case(B=B, S=S, N=N, C=C, k=k, seed=131, wstd=0.3)
    rng = np.random.default_rng(4)
    W_pp = rng.standard_normal((N + 4 * k, N * C)) * 0.3
    W_ra = rng.standard_normal((k * k, k * C)) * 0.3
    dXp = rng.standard_normal(X.shape)
    g = xo.backward(X, out, cv, xo.expand_hres_active(W_pp, W_ra, idx, N, C), idx, dXp)
    dW_ra = xo.gather_hres_active(g["dW"], idx, N, C)

    def L():
        return (xo.forward(X, out, cv, xo.expand_hres_active(W_pp, W_ra, idx, N, C), idx)["Xp"] * dXp).sum()

    num, _ = fd(L, W_ra)
    np.testing.assert_allclose(dW_ra, num, rtol=1e-6, atol=1e-8)
