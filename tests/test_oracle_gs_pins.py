"""Pins of the oracle's modified Gram-Schmidt of the TFA components.

Source: "xHC: Expanded Hyper-Connections" (qingkeai.online), section
"Conv / Gram-Schmidt": the raw output u_0 is kept and each convolution
component has its projections onto the components before it removed one at a
time, so that the four write-back features are mutually orthogonal.

Each test checks the oracle against something other than itself: the QR
factorisation of a library routine (Gram-Schmidt of the rows of U is U^T = QR
with u~_c = R[c, c] Q[:, c]), orthogonality and span invariants, special
cases with a known answer, and central finite differences of the backward.
"""
import numpy as np
import pytest

from oracle import xhc_oracle as xo
from tests.test_oracle_pins import case, fd


def _rows(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_gs_equals_qr_columns_times_diagonal():
    u = _rows((4, 6, 9), 1)
    ut, _ = xo.gram_schmidt(u)
    for s in range(u.shape[1]):
        Q, R = np.linalg.qr(u[:, s, :].T)          # [C, 4], [4, 4]
        ref = (Q * np.diag(R)[None, :]).T          # row c = R[c, c] Q[:, c]
        np.testing.assert_allclose(ut[:, s, :], ref, rtol=0, atol=1e-12)


def test_gs_orthogonal_and_triangular():
    u = _rows((4, 5, 16), 2)
    u[1] += 0.9 * u[0]                             # strongly correlated, as the pages report
    u[3] += 0.7 * u[1] - 0.5 * u[2]
    ut, _ = xo.gram_schmidt(u)
    np.testing.assert_array_equal(ut[0], u[0])
    g = np.einsum("asc,bsc->sab", ut, ut)
    scale = np.sqrt(np.einsum("saa->sa", g))
    off = g / (scale[:, :, None] * scale[:, None, :])
    off[:, np.arange(4), np.arange(4)] = 0.0
    assert np.abs(off).max() < 1e-13
    # u_c - u~_c lies in the span of u_0 .. u_{c-1}
    for s in range(u.shape[1]):
        for c in range(1, 4):
            A = u[:c, s, :].T
            r = u[c, s] - ut[c, s]
            coef, *_ = np.linalg.lstsq(A, r, rcond=None)
            assert np.linalg.norm(A @ coef - r) <= 1e-12 * max(1.0, np.linalg.norm(r))


def test_gs_identity_on_orthogonal_rows():
    base = _rows((7, 4), 3)
    Q, _ = np.linalg.qr(base)                      # orthonormal columns
    u = np.stack([Q[:, c] * (c + 2.0) for c in range(4)])[:, None, :]
    ut, _ = xo.gram_schmidt(u)
    np.testing.assert_allclose(ut, u, rtol=0, atol=1e-14)


def test_gs_zero_components_are_skipped():
    u = _rows((4, 3, 8), 4)
    u[2] = 0.0
    ut, _ = xo.gram_schmidt(u)
    assert np.all(ut[2] == 0.0)
    # u~_3 is the third output of Gram-Schmidt over (u_0, u_1, u_3)
    ref, _ = xo.gram_schmidt(np.stack([u[0], u[1], u[3], np.zeros_like(u[0])]))
    np.testing.assert_allclose(ut[3], ref[2], rtol=0, atol=1e-13)
    # a zero u_0 removes nothing from the later components
    v = _rows((4, 2, 8), 5)
    v[0] = 0.0
    vt, _ = xo.gram_schmidt(v)
    np.testing.assert_array_equal(vt[1], v[1])


def test_gs_without_convolutions_changes_nothing():
    X, out, _, W, idx = case(B=1, S=6, N=16, C=8, seed=7, conv=False)
    a = xo.forward(X, out, None, W, idx)
    b = xo.forward(X, out, None, W, idx, gs=True)
    np.testing.assert_array_equal(a["Xp"], b["Xp"])


def test_gs_changes_the_write_when_components_correlate():
    X, out, cv, W, idx = case(B=1, S=10, N=16, C=8, seed=8, cstd=0.6)
    a = xo.forward(X, out, cv, W, idx)
    b = xo.forward(X, out, cv, W, idx, gs=True)
    assert np.abs(a["Xp"] - b["Xp"]).max() > 1e-3
    inactive = [n for n in range(16) if n not in idx]
    np.testing.assert_array_equal(b["Xp"][:, :, inactive], X[:, :, inactive])


def test_gs_reverse_finite_differences():
    u = _rows((4, 3, 5), 9)
    u[2] += 0.8 * u[1]
    R = _rows((4, 3, 5), 10)
    ut, steps = xo.gram_schmidt(u)
    du = xo.gram_schmidt_reverse(R, ut, steps)
    L = lambda: float((xo.gram_schmidt(u)[0] * R).sum())
    num, _ = fd(L, u)
    np.testing.assert_allclose(du, num, rtol=1e-7, atol=1e-8)


@pytest.mark.parametrize("with_dxin", [False, True])
def test_gs_backward_finite_differences(with_dxin):
    B, S, C = 1, 14, 3
    X, out, cv, W, idx = case(B=B, S=S, N=16, C=C, k=4, seed=120, wstd=0.3, cstd=0.5)
    rng = np.random.default_rng(11)
    dXp = rng.standard_normal(X.shape)
    dxi = rng.standard_normal(out.shape) if with_dxin else None
    g = xo.backward(X, out, cv, W, idx, dXp, dxi, gs=True)

    def L():
        r = xo.forward(X, out, cv, W, idx, gs=True)
        val = (r["Xp"] * dXp).sum()
        if dxi is not None:
            val += (r["x_in"] * dxi).sum()
        return val

    num, _ = fd(L, out)
    np.testing.assert_allclose(g["dout"], num, rtol=1e-6, atol=1e-7)
    for w, dw in zip(cv, g["dconv"]):
        num, _ = fd(L, w)
        np.testing.assert_allclose(dw, num, rtol=1e-6, atol=1e-7)
    picks = [tuple(rng.integers(0, s) for s in X.shape) for _ in range(30)]
    num, it = fd(L, X, picks=picks)
    for ix in it:
        assert abs(num[ix] - g["dX"][ix]) <= 1e-6 * max(1.0, abs(num[ix])), ix
    picks = [tuple(rng.integers(0, s) for s in W.shape) for _ in range(30)]
    num, it = fd(L, W, picks=picks)
    for ix in it:
        assert abs(num[ix] - g["dW"][ix]) <= 1e-6 * max(1.0, abs(num[ix])), ix


def test_gs_dependent_component_is_skipped():
    # u_2 in the span of u_0, u_1: its residual vanishes (relative to |u_2|)
    # and nothing is projected onto it
    u = _rows((4, 3, 8), 12)
    u[2] = 2.0 * u[1] - u[0]
    ut, steps = xo.gram_schmidt(u)
    assert np.abs(ut[2]).max() < 1e-12 * np.abs(u[2]).max()
    assert not any(st[5].any() for st in steps if st[1] == 2)
    ref, _ = xo.gram_schmidt(np.stack([u[0], u[1], u[3], np.zeros_like(u[0])]))
    np.testing.assert_allclose(ut[3], ref[2], rtol=0, atol=1e-12)
