"""Pins of the oracle's stack of sublayers (forward_stack) and of its bf16
state rounding (round_bf16).

Source: "xHC: Expanded Hyper-Connections" (qingkeai.online), sections "Dense
read, sparse write" (sublayer l + 1 reads the state that sublayer l scattered
its k rows into) and "Beyond N=16" (xHC-Flash: the stack's traffic is lowered
by reordering reads and writes, and the dense-read correction over the k
changed rows is exact).

Each test checks the stack against something other than the stack itself:
bf16 rounding against ties worked by hand and against the integer bit rule;
the next sublayer's logits and dense read against the xHC-Flash correction
identities computed from the states alone; a closed form with W = 0 and zero
convolutions; and locality of a perturbed output.
"""
import numpy as np

from oracle import xhc_oracle as xo
from tests.test_oracle_pins import case


def _stack_case(L, B=2, S=14, N=16, C=5, k=4, seed=300, wstd=0.3, same_idx=False):
    X, *_ = case(B=B, S=S, N=N, C=C, k=k, seed=seed, wstd=wstd)
    outs, convs, Ws, idxs = [], [], [], []
    for l in range(L):
        _, out, cv, W, idx = case(B=B, S=S, N=N, C=C, k=k, seed=seed + 10 * (l + 1), wstd=wstd)
        outs.append(out)
        convs.append(cv)
        Ws.append(W)
        idxs.append(idxs[0] if (same_idx and l) else idx)
    return X, outs, convs, Ws, idxs


def test_round_bf16_ties_and_bit_rule():
    # ties worked by hand: the bf16 spacing at 1 is 2^-7
    assert xo.round_bf16(1 + 2.0 ** -8) == 1.0                          # tie, even mantissa below
    assert xo.round_bf16(1 + 3 * 2.0 ** -8) == 1 + 2.0 ** -6            # tie, even mantissa above
    assert xo.round_bf16(-(1 + 3 * 2.0 ** -8)) == -(1 + 2.0 ** -6)
    assert xo.round_bf16(1 + 2.0 ** -8 + 2.0 ** -20) == 1 + 2.0 ** -7   # just above the tie
    assert xo.round_bf16(0.0) == 0.0
    # float32 inputs: the integer rule (add 0x7FFF plus the kept lowest bit, drop 16 bits)
    a = np.random.default_rng(301).standard_normal(20000).astype(np.float32) * 7
    u = a.view(np.uint32).astype(np.uint64)
    bits = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    ref = bits.astype(np.uint32).view(np.float32).astype(np.float64)
    np.testing.assert_array_equal(xo.round_bf16(a.astype(np.float64)), ref)


def test_one_sublayer_is_the_update():
    X, outs, convs, Ws, idxs = _stack_case(1, seed=310)
    r = xo.forward_stack(X, outs, convs, Ws, idxs)
    # the plain update of X written out by hand for one token
    f = xo.forward(X, outs[0], convs[0], Ws[0], idxs[0])
    np.testing.assert_array_equal(r["states"][1], f["Xp"])
    np.testing.assert_array_equal(r["x_in"][0], f["x_in"])
    np.testing.assert_array_equal(r["states"][0], X)


def test_next_sublayer_from_the_correction_identities():
    """xHC-Flash: sublayer l + 1's logits and dense read follow from the state
    before sublayer l and the k rows it changed:
      p_{l+1} = vec S_l W^T + sum_i (S_{l+1}[a_i] - S_l[a_i]) W[:, a_i block]^T
      ss_{l+1} = |vec S_l|^2 + sum_i (|S_{l+1}[a_i]|^2 - |S_l[a_i]|^2)
      x_in_{l+1} = sum_n hpre[n] S_l[n] + sum_i hpre[a_i] (S_{l+1}[a_i] - S_l[a_i])
    checked against the stack's own sublayer l + 1, with and without bf16
    storage between sublayers."""
    X, outs, convs, Ws, idxs = _stack_case(3, seed=320)
    B, S, N, C = X.shape
    eps = 1e-6
    for store in (None, "bf16"):
        # a bf16 state starts from bf16 values
        X0 = xo.round_bf16(X) if store else X
        r = xo.forward_stack(X0, outs, convs, Ws, idxs, eps=eps, store=store)
        for l in range(2):
            Sl, Sn, W, a = r["states"][l + 1], r["states"][l + 2], Ws[l + 1], [int(i) for i in idxs[l]]
            Sprev = r["states"][l]
            # sublayer l + 1 reads states[l + 1]: states[l] plus the k rows sublayer l wrote
            D = Sl[:, :, a, :] - Sprev[:, :, a, :]                       # [B, S, k, C]
            v = Sprev.reshape(B, S, N * C)
            p = v @ W.T
            for i, n in enumerate(a):
                p += D[:, :, i, :] @ W[:, n * C:(n + 1) * C].T
            ss = (v * v).sum(axis=2) + ((Sl[:, :, a, :] ** 2) - (Sprev[:, :, a, :] ** 2)).sum(axis=(2, 3))
            z = p / np.sqrt(ss / (N * C) + eps)[:, :, None]
            np.testing.assert_allclose(z, r["z"][l + 1], rtol=1e-11, atol=1e-11)
            hpre = 1.0 / (1.0 + np.exp(-z[:, :, :N]))
            x = np.einsum("bsn,bsnc->bsc", hpre, Sprev)
            for i, n in enumerate(a):
                x += hpre[:, :, n, None] * D[:, :, i, :]
            np.testing.assert_allclose(x, r["x_in"][l + 1], rtol=1e-11, atol=1e-11)
            assert Sn.shape == Sl.shape


def test_zero_weights_closed_form():
    """W = 0 and zero convolutions: every sublayer sets its active rows to
    the mean of their previous values plus out_l / 2 (H^res = J/k, H^post =
    1/2, u_1..u_3 = 0), and its dense read is half the sum of the streams."""
    L, B, S, N, C, k = 3, 2, 9, 16, 4, 4
    X, outs, convs, Ws, _ = _stack_case(L, B=B, S=S, N=N, C=C, k=k, seed=330)
    Ws = [np.zeros_like(W) for W in Ws]
    convs = [tuple(np.zeros_like(w) for w in cv) for cv in convs]
    a, b = [3, 7, 1, 12], [5, 0, 9, 14]                  # disjoint sets
    idxs = [a, b, a]
    r = xo.forward_stack(X, outs, convs, Ws, idxs)
    ref = X.copy()
    for l, ix in enumerate(idxs):
        np.testing.assert_allclose(r["x_in"][l], 0.5 * ref.sum(axis=2), rtol=1e-13, atol=1e-13)
        m = ref[:, :, ix, :].mean(axis=2)
        for n in ix:
            ref[:, :, n, :] = m + 0.5 * outs[l]
    np.testing.assert_allclose(r["states"][-1], ref, rtol=1e-13, atol=1e-13)
    # rows of b were written once (sublayer 1), rows of a twice (sublayers 0 and 2)
    np.testing.assert_allclose(r["states"][-1][:, :, b[0]], X[:, :, b, :].mean(axis=2) + 0.5 * outs[1],
                               rtol=1e-13, atol=1e-13)
    untouched = [n for n in range(N) if n not in a + b]
    np.testing.assert_array_equal(r["states"][-1][:, :, untouched], X[:, :, untouched])


def test_perturbed_output_stays_in_its_halo():
    """A change of out_l at token t of one sequence moves the final state only
    at tokens t .. t + 11 of that sequence: later sublayers act on each token
    separately and read only their own outputs."""
    X, outs, convs, Ws, idxs = _stack_case(3, B=2, S=30, seed=340)
    base = xo.forward_stack(X, outs, convs, Ws, idxs)["states"][-1]
    outs2 = [o.copy() for o in outs]
    t = 9
    outs2[1][1, t, :] += 0.5
    got = xo.forward_stack(X, outs2, convs, Ws, idxs)["states"][-1]
    changed = np.nonzero(np.abs(got - base).max(axis=(2, 3)) > 0)
    assert set(changed[0]) == {1}
    assert set(changed[1]) <= set(range(t, t + 12)) and t in set(changed[1])
    np.testing.assert_array_equal(got[0], base[0])
    np.testing.assert_array_equal(got[1, :t], base[1, :t])
