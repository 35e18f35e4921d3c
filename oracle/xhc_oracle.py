"""Plain fp64 CPU oracle of the xHC per-sublayer residual-stream update.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this module:
it is used by ``tests/``, by ``__graft_entry__.smoke()`` (to check one small GPU
run) and by ``bench.py``'s ``cpu_baseline`` / ``--impl reference`` legs.  It
shares no code with the CUDA library under ``residual_stream_expansion_xhc_b300``.

Sources (page, section), from "xHC: Expanded Hyper-Connections" (qingkeai.online
research retrospective, cited below as [xHC]):

* [xHC] "Scaling N": the state of a sublayer is N residual streams of width C;
  H^pre reads the sublayer input from the streams, H^post writes the output
  back, H^res mixes the streams and is made doubly stochastic by Sinkhorn.
* [xHC] "Write-back bottleneck": the mHC write of stream i is h^post_i * out.
* [xHC] "Temporal Feature Augmentation": out in R^{S x C}; three causal
  depthwise convolutions with kernel sizes 4, 8, 12 along the sequence, each
  channel on its own, stacked with the raw output into 4 components.
* [xHC] "Conv / Gram-Schmidt": the components u_c in R^C, c = 0..3.
* [xHC] "Dense read, sparse write": the sublayer input is read from all N
  streams; only the k active streams (set A_l, |A_l| = k) are written, by a
  combination sum_c h^post_{l,i,c} u_c; inactive streams are left unchanged
  and only the active streams take part in the H^res mixing.

The formulas themselves did not survive on the pages; the formulation below is
the one fixed by the project specification, with these readings where the
pages are silent (each is listed in the design notes):

* rmsnorm over the whole flattened state vec X (length N*C), eps = 1e-6, no
  gain; projection W of shape [P, N*C], P = N + 4k + k^2, no bias.
* rows of W: [0, N) -> H^pre; N + 4i + c -> H^post[i, c];
  N + 4k + k*i + j -> H^res logit [i, j]; W's columns follow vec X's order
  n*C + c.
* H^pre, H^post: plain sigmoid.  H^res: exp(Z - max Z), then ``iters`` times
  (normalise rows, then normalise columns).
* X'[a_i] = sum_j H^res[i, j] X[a_j] + sum_c H^post[i, c] u_c for slot i of
  the ordered index list a; other streams unchanged.
* conv tap tau multiplies out[t - tau] (tau = 0 is the current token), zero
  padding before the start of each sequence, no bias.  Router score s = 1 (the
  active indices are given).
* Gram-Schmidt ([xHC] "Conv / Gram-Schmidt"; optional, ``gs=True``): per token,
  modified Gram-Schmidt over the four components in the order u_0, u_1, u_2,
  u_3: u~_0 = u_0 is kept, and each later component has its projections onto
  the earlier u~_d removed one at a time, each projection taken from the
  partly reduced vector.  The write-back then combines u~_c instead of u_c.
  The pages leave a zero (or vanishing) component undefined; reading: a
  projection onto u~_d is skipped (its coefficient taken as 0) when
  |u~_d|^2 <= GS_EPS |u_d|^2, i.e. when u_d is zero or lies (to within a
  relative 1e-3 in norm) in the span of the components before it.  A zero
  component then stays zero and removes nothing.

All arrays are float64 numpy arrays.  The backward is the exact reverse mode of
the forward, hand-derived step by step (the Sinkhorn reverse recomputes and
keeps the forward iterates).  Sequences are processed one at a time to bound
memory; nothing couples two sequences except the weight-gradient sums.
"""
from __future__ import annotations

import numpy as np

CONV_KS = (4, 8, 12)
GS_EPS = 1e-6       # relative squared residual at or below which a component is treated as zero


def n_logits(N: int, k: int) -> int:
    """P = N (H^pre) + 4k (H^post) + k^2 (H^res logits)."""
    return N + 4 * k + k * k


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def sinkhorn(Z, iters):
    """exp(Z - max Z) followed by ``iters`` rounds of (row-normalise,
    column-normalise), batched over leading axes.  Z: [..., k, k].

    Returns (H, trace) where trace keeps every intermediate matrix for the
    reverse pass: trace[0] = M0 = exp(Z - max Z); then for each iteration the
    matrix before the row step and before the column step.
    """
    zmax = Z.max(axis=(-2, -1), keepdims=True)
    M = np.exp(Z - zmax)
    trace = [M]
    for _ in range(iters):
        before_row = M
        M = M / M.sum(axis=-1, keepdims=True)      # row i: sum over j
        before_col = M
        M = M / M.sum(axis=-2, keepdims=True)      # column j: sum over i
        trace.append((before_row, before_col))
    return M, trace


def sinkhorn_reverse(dH, trace):
    """Reverse mode of ``sinkhorn``: given dL/dH, return dL/dZ.

    A normalisation y = x / s with s = sum over the normalised axis of x has
    dL/dx = dL/dy / s - sum_axis(dL/dy * x) / s^2 (broadcast along the axis).
    The max subtracted before exp is treated as a constant: a shift of one
    row's logits is removed exactly by the next row normalisation, so its
    gradient contribution is zero.
    """
    g = dH
    for before_row, before_col in reversed(trace[1:]):
        s = before_col.sum(axis=-2, keepdims=True)
        g = g / s - (g * before_col).sum(axis=-2, keepdims=True) / (s * s)
        s = before_row.sum(axis=-1, keepdims=True)
        g = g / s - (g * before_row).sum(axis=-1, keepdims=True) / (s * s)
    M0 = trace[0]
    return g * M0


def tfa_components(out_seq, conv):
    """Temporal Feature Augmentation of one sequence.

    out_seq: [S, C].  conv: (w4 [C,4], w8 [C,8], w12 [C,12]) or None.
    Returns u: [4, S, C] with u[0] = out and u[j][t, c] =
    sum_{tau < K_j} w_j[c, tau] * out[t - tau, c] (zero for t - tau < 0).
    With conv = None the three convolution components are zero.
    """
    S, C = out_seq.shape
    u = np.zeros((4, S, C))
    u[0] = out_seq
    if conv is None:
        return u
    for j, w in enumerate(conv, start=1):
        K = w.shape[1]
        for tau in range(K):
            if tau >= S:
                break
            # u_j[t] += w[:, tau] * out[t - tau] for t >= tau
            u[j, tau:, :] += w[None, :, tau] * out_seq[: S - tau, :]
    return u


def gram_schmidt(u, eps=GS_EPS):
    """Modified Gram-Schmidt of the four components of every token.

    u: [4, S, C] (component, token, channel).  Returns (ut, steps): ut[0] =
    u[0]; for c = 1, 2, 3 the vector v starts as u[c] and, for d = 0 .. c-1 in
    turn, loses its projection onto ut[d]:
        alpha = <v, ut[d]> / <ut[d], ut[d]>   (0 when <ut[d], ut[d]> <= eps <u_d, u_d>)
        v    <- v - alpha ut[d]
    and ut[c] is the final v.  ``steps`` keeps, per (c, d), the vector before
    the step, alpha, the squared norm and the skip mask for the reverse pass.
    """
    ut = np.empty_like(u)
    ut[0] = u[0]
    raw = np.einsum("xsc,xsc->xs", u, u)
    norms = [raw[0]]
    steps = []
    for c in range(1, 4):
        v = u[c].copy()
        for d in range(c):
            n = norms[d]
            use = n > eps * raw[d]
            alpha = np.where(use, np.einsum("sc,sc->s", v, ut[d]) / np.where(use, n, 1.0), 0.0)
            steps.append((c, d, v.copy(), alpha, n, use))
            v = v - alpha[:, None] * ut[d]
        ut[c] = v
        norms.append(np.einsum("sc,sc->s", v, v))
    return ut, steps


def gram_schmidt_reverse(dut, ut, steps):
    """Reverse mode of ``gram_schmidt``: dL/dut [4, S, C] -> dL/du.

    Steps are undone last to first.  For v' = v - alpha ut_d with alpha =
    <v, ut_d> / n_d and n_d = <ut_d, ut_d> (the skip decision is a constant):
        dL/dalpha = -<g, ut_d>
        dL/dv    += g + dL/dalpha ut_d / n_d
        dL/dut_d += -alpha g + dL/dalpha (v / n_d - 2 alpha ut_d / n_d)
    where g = dL/dv'.
    """
    acc = dut.copy()                  # dL/dut, growing as later steps are undone
    du = np.zeros_like(dut)
    by_c = {}
    for st in steps:
        by_c.setdefault(st[0], []).append(st)
    for c in (3, 2, 1):
        g = acc[c].copy()             # dL/d(final v of component c)
        for (_, d, v, alpha, n, use) in reversed(by_c[c]):
            da = -np.einsum("sc,sc->s", g, ut[d])
            inv = np.where(use, 1.0 / np.where(use, n, 1.0), 0.0)
            acc[d] += (-alpha[:, None] * g
                       + (da * inv)[:, None] * v
                       - (2.0 * da * alpha * inv)[:, None] * ut[d])
            g = g + (da * inv)[:, None] * ut[d]
        du[c] = g
    du[0] = acc[0]
    return du


def _check(X, out, conv, W, idx):
    B, S, N, C = X.shape
    k = len(idx)
    assert out.shape == (B, S, C)
    assert W.shape == (n_logits(N, k), N * C)
    assert len(set(int(a) for a in idx)) == k and all(0 <= int(a) < N for a in idx)
    if conv is not None:
        assert tuple(w.shape for w in conv) == tuple((C, K) for K in CONV_KS)
    return B, S, N, C, k


def _coeffs_seq(Xs, W, N, C, k, iters, eps):
    """Coefficients for one sequence.  Xs: [S, N, C]."""
    S = Xs.shape[0]
    v = Xs.reshape(S, N * C)
    rstd = 1.0 / np.sqrt((v * v).mean(axis=1) + eps)           # rmsnorm scale
    p = v @ W.T                                                  # [S, P]
    z = rstd[:, None] * p
    hpre = sigmoid(z[:, :N])
    hpost = sigmoid(z[:, N:N + 4 * k]).reshape(S, k, 4)
    Z = z[:, N + 4 * k:].reshape(S, k, k)
    hres, trace = sinkhorn(Z, iters)
    return dict(v=v, rstd=rstd, p=p, z=z, hpre=hpre, hpost=hpost, hres=hres, trace=trace)


def forward(X, out, conv, W, idx, iters=20, eps=1e-6, gs=False):
    """One xHC sublayer update (forward).

    X: [B, S, N, C]; out: [B, S, C]; conv: (w4, w8, w12) or None;
    W: [P, N*C]; idx: the k active stream indices (ordered, slot i <-> idx[i]);
    gs: orthogonalise the components by modified Gram-Schmidt first.

    Returns a dict with Xp (updated state [B,S,N,C]), x_in (dense read
    [B,S,C]), z (logits [B,S,P]), rstd [B,S], hpre [B,S,N], hpost [B,S,k,4],
    hres [B,S,k,k], u (the components written back, after Gram-Schmidt when
    gs, [B,4,S,C]).
    """
    B, S, N, C, k = _check(X, out, conv, W, idx)
    idx = [int(a) for a in idx]
    P = n_logits(N, k)
    res = dict(Xp=X.copy(), x_in=np.zeros((B, S, C)), z=np.zeros((B, S, P)),
               rstd=np.zeros((B, S)), hpre=np.zeros((B, S, N)),
               hpost=np.zeros((B, S, k, 4)), hres=np.zeros((B, S, k, k)),
               u=np.zeros((B, 4, S, C)))
    for b in range(B):
        cf = _coeffs_seq(X[b], W, N, C, k, iters, eps)
        # dense read over all N streams
        x_in = np.einsum("sn,snc->sc", cf["hpre"], X[b])
        u = tfa_components(out[b], conv)
        if gs:
            u, _ = gram_schmidt(u)
        Xa = X[b][:, idx, :]                                     # [S, k, C]
        mix = np.einsum("sij,sjc->sic", cf["hres"], Xa)
        write = np.einsum("sic,csx->six", cf["hpost"], u)       # sum over components
        res["Xp"][b][:, idx, :] = mix + write
        res["x_in"][b] = x_in
        res["u"][b] = u
        for key in ("z", "rstd", "hpre", "hpost", "hres"):
            res[key][b] = cf[key]
    return res


def round_bf16(x):
    """Nearest bf16 value of each entry (round half to even), as float64.

    A bf16 number keeps 8 significant bits: x = m 2^e with 1/2 <= |m| < 1 is
    replaced by round(m 2^8) 2^(e - 8).  Magnitudes stay far inside bf16's
    exponent range here, so neither overflow nor subnormals arise.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.round(np.ldexp(m, 8)), e - 8)


def forward_stack(X, outs, convs, Ws, idxs, iters=20, eps=1e-6, gs=False, store=None):
    """A stack of L sublayers applied in order to one state (in place in
    memory): sublayer l reads the state S_l that sublayer l - 1 wrote, with its
    own out_l, conv_l, W_l and index list a_l, and writes S_{l+1}.

    [xHC] "Dense read, sparse write" (the state of the next sublayer is the
    scatter-updated state of this one; the next input is a dense read of it)
    and "Beyond N=16" (xHC-Flash: a stack whose per-sublayer memory traffic a
    reordered schedule lowers, with an exact dense-read correction).  ``store="bf16"``: the state is rounded to bf16 after
    every sublayer, as a bf16 state in memory holds it between sublayers; the
    first state is taken as given.

    Returns dict(states=[S_0 .. S_L], x_in=[per sublayer], z=[per sublayer],
    rstd=[per sublayer]).
    """
    L = len(outs)
    assert len(convs) == len(Ws) == len(idxs) == L
    states, x_ins, zs, rstds = [X], [], [], []
    S = X
    for l in range(L):
        r = forward(S, outs[l], convs[l], Ws[l], idxs[l], iters=iters, eps=eps, gs=gs)
        S = round_bf16(r["Xp"]) if store == "bf16" else r["Xp"]
        states.append(S)
        x_ins.append(r["x_in"])
        zs.append(r["z"])
        rstds.append(r["rstd"])
    return dict(states=states, x_in=x_ins, z=zs, rstd=rstds)


def backward(X, out, conv, W, idx, dXp, dx_in=None, iters=20, eps=1e-6, keep=False, gs=False):
    """Exact reverse mode of ``forward``.

    X is the state BEFORE the update.  dXp = dL/dX' [B,S,N,C]; dx_in = dL/dx_in
    [B,S,C] or None (no gradient through the dense read).

    Returns dict with dX [B,S,N,C], dout [B,S,C], dconv (three arrays, or None
    when conv is None), dW [P, N*C]; with keep=True also dz [B,S,P] (gradient
    at the logits) and the per-token dp [B,S,P] and drstd [B,S].  gs: the
    forward orthogonalised the components (``gram_schmidt``); the gradient
    at the orthogonalised components is taken back through it.
    """
    B, S, N, C, k = _check(X, out, conv, W, idx)
    idx = [int(a) for a in idx]
    inactive = [n for n in range(N) if n not in idx]
    P = n_logits(N, k)
    dX = np.zeros_like(X)
    dout = np.zeros_like(out)
    dW = np.zeros_like(W)
    dconv = None if conv is None else [np.zeros_like(w) for w in conv]
    extra = dict(dz=np.zeros((B, S, P)), dp=np.zeros((B, S, P)), drstd=np.zeros((B, S)))
    for b in range(B):
        Xs = X[b]
        cf = _coeffs_seq(Xs, W, N, C, k, iters, eps)
        u = tfa_components(out[b], conv)                        # [4, S, C]
        if gs:
            u_raw = u
            u, gs_steps = gram_schmidt(u_raw)
        G = dXp[b][:, idx, :]                                   # [S, k, C]
        Xa = Xs[:, idx, :]                                      # [S, k, C]
        # gradients at the coefficients
        d_hres = np.einsum("sic,sjc->sij", G, Xa)
        d_hpost = np.einsum("sic,xsc->six", G, u)
        if dx_in is not None:
            d_hpre = np.einsum("sc,snc->sn", dx_in[b], Xs)
        else:
            d_hpre = np.zeros((S, N))
        # through the nonlinearities to the logits
        dZ = sinkhorn_reverse(d_hres, cf["trace"])             # [S, k, k]
        hpre, hpost = cf["hpre"], cf["hpost"]
        dz = np.concatenate([
            d_hpre * hpre * (1.0 - hpre),
            (d_hpost * hpost * (1.0 - hpost)).reshape(S, 4 * k),
            dZ.reshape(S, k * k)], axis=1)
        # z = rstd * p
        rstd, p, v = cf["rstd"], cf["p"], cf["v"]
        dp = rstd[:, None] * dz
        drstd = (dz * p).sum(axis=1)
        # p = W v ;  rstd = (mean(v^2) + eps)^(-1/2)  => d rstd / dv = -rstd^3 v / (N C)
        dv = dp @ W + (drstd * (-(rstd ** 3) / (N * C)))[:, None] * v
        dW += dp.T @ v
        dXs = dv.reshape(S, N, C).copy()
        # dense read x_in = sum_n hpre[n] X[n]
        if dx_in is not None:
            dXs += hpre[:, :, None] * dx_in[b][:, None, :]
        # sparse write: inactive streams pass through, active ones are mixed
        dXs[:, inactive, :] += dXp[b][:, inactive, :]
        dXs[:, idx, :] += np.einsum("sij,sic->sjc", cf["hres"], G)
        dX[b] = dXs
        # components: du_c = sum_i hpost[i, c] G_i
        du = np.einsum("six,sic->xsc", hpost, G)                # [4, S, C]
        if gs:
            du = gram_schmidt_reverse(du, u, gs_steps)
        dout_b = du[0].copy()
        if conv is not None:
            for j, w in enumerate(conv, start=1):
                K = w.shape[1]
                for tau in range(min(K, S)):
                    # u_j[t] += w[:, tau] * out[t - tau]  (t >= tau)
                    dout_b[: S - tau, :] += w[None, :, tau] * du[j, tau:, :]
                    dconv[j - 1][:, tau] += (du[j, tau:, :] * out[b][: S - tau, :]).sum(axis=0)
        dout[b] = dout_b
        extra["dz"][b] = dz
        extra["dp"][b] = dp
        extra["drstd"][b] = drstd
    res = dict(dX=dX, dout=dout, dconv=dconv, dW=dW)
    if keep:
        res.update(extra)
    return res


def expand_hres_active(W_pp, W_ra, idx, N, C):
    """H^res logits from the k active streams only ([xHC] "Dense read, sparse
    write": only the active streams take part in the residual mixing, so the
    mixing logits need only their k*C entries -- the O(k^3 C) reading).

    W_pp: [N + 4k, N*C] (H^pre and H^post rows over the whole state);
    W_ra: [k*k, k*C] (H^res rows over vec(X[a_0], ..., X[a_{k-1}]), slot
    order).  Returns the full projection [P, N*C] whose H^res rows carry W_ra
    in the columns of the active streams and zeros elsewhere, so that
    z_res = rstd * vec(X_A) . W_ra^T through the plain forward.
    """
    k = len(idx)
    W = np.zeros((N + 4 * k + k * k, N * C))
    W[: N + 4 * k] = W_pp
    for j, a in enumerate(idx):
        W[N + 4 * k:, int(a) * C:(int(a) + 1) * C] = W_ra[:, j * C:(j + 1) * C]
    return W


def gather_hres_active(dW, idx, N, C):
    """dL/dW_ra from dL/dW of the expanded projection: the active streams'
    columns of the H^res rows, in slot order."""
    k = len(idx)
    return np.concatenate([dW[N + 4 * k:, int(a) * C:(int(a) + 1) * C] for a in idx], axis=1)


# ---------------------------------------------------------------- router with per-token active sets
#
# [xHC] "Dense read, sparse write": the router reads the LayerNorm-ed whole
# state vec X and gives every stream a sigmoid score; some streams are always
# active (fixed) and the others are chosen per token by top-k of the scores.
# For a chosen (routed) stream the score multiplies that stream's new
# write-back, so the router learns through the write-back's size; unchosen
# scores get no gradient in this sublayer.  Readings (the pages give no
# formulas): LayerNorm over all N*C entries without gain or bias, eps as the
# rmsnorm's; router weights W_r [N, N*C], no bias; the fixed streams are a
# caller-given ordered list and take the first slots; the routed slots follow
# in descending score (ties to the lower stream index); H^post and H^res rows
# belong to slots as in the plain update.


def router_scores(Xs, W_r, eps):
    """Scores of one sequence.  Xs [S, N, C], W_r [N, N*C].  Returns
    (s [S, N] sigmoid scores, r [S, N] logits, y [S, N*C] LayerNorm-ed state,
    sd [S] its standard deviation sqrt(var + eps))."""
    S, N, C = Xs.shape
    v = Xs.reshape(S, N * C)
    mu = v.mean(axis=1)
    sd = np.sqrt(((v - mu[:, None]) ** 2).mean(axis=1) + eps)
    y = (v - mu[:, None]) / sd[:, None]
    r = y @ W_r.T
    return sigmoid(r), r, y, sd


def route(scores, fixed, k):
    """Per-token active slots: the fixed streams in the given order, then the
    top (k - len(fixed)) other streams by score (descending, ties to the lower
    index).  scores [S, N] -> idx [S, k] (int)."""
    S, N = scores.shape
    fixed = [int(a) for a in fixed]
    others = [n for n in range(N) if n not in fixed]
    idx = np.zeros((S, k), dtype=np.int64)
    for t in range(S):
        order = sorted(others, key=lambda n: (-scores[t, n], n))
        idx[t] = fixed + order[: k - len(fixed)]
    return idx


def _routed_weights(s, idx, nfixed):
    """w[t, i] = 1 for fixed slots, the routed stream's score otherwise."""
    w = np.take_along_axis(s, idx, axis=1).copy()
    w[:, :nfixed] = 1.0
    return w


def forward_routed(X, out, conv, W, W_r, fixed, k, iters=20, eps=1e-6, idx=None):
    """The sublayer update with per-token active sets chosen by the router.
    X [B,S,N,C], out [B,S,C], conv as in ``forward``, W [P, N*C] (P for k
    slots), W_r [N, N*C], fixed: the always-active streams (ordered).
    ``idx`` [B, S, k] optionally gives the active sets (where two scores tie
    either choice is a valid forward); by default ``route`` chooses them.
    Returns Xp, x_in, idx [B,S,k], s [B,S,N]."""
    B, S, N, C = X.shape
    res = dict(Xp=X.copy(), x_in=np.zeros((B, S, C)), idx=np.zeros((B, S, k), dtype=np.int64),
               s=np.zeros((B, S, N)))
    for b in range(B):
        cf = _coeffs_seq(X[b], W, N, C, k, iters, eps)
        s, _, _, _ = router_scores(X[b], W_r, eps)
        ib = route(s, fixed, k) if idx is None else np.asarray(idx[b], dtype=np.int64)
        w = _routed_weights(s, ib, len(fixed))
        u = tfa_components(out[b], conv)
        Xa = np.take_along_axis(X[b], ib[:, :, None], axis=1)               # [S, k, C]
        mix = np.einsum("sij,sjc->sic", cf["hres"], Xa)
        write = np.einsum("sic,csx->six", cf["hpost"], u) * w[:, :, None]
        Xp = X[b].copy()
        np.put_along_axis(Xp, ib[:, :, None], mix + write, axis=1)
        res["Xp"][b] = Xp
        res["x_in"][b] = np.einsum("sn,snc->sc", cf["hpre"], X[b])
        res["idx"][b] = ib
        res["s"][b] = s
    return res


def backward_routed(X, out, conv, W, W_r, fixed, k, dXp, dx_in=None, iters=20, eps=1e-6, idx=None):
    """Exact reverse mode of ``forward_routed`` (the active sets are the
    forward's, a constant; unchosen scores get no gradient).  ``idx``
    [B, S, k] optionally gives the active sets (where two scores tie either
    choice is a valid forward); by default ``route`` chooses them.  Returns
    dX, dout, dconv, dW, dW_r."""
    B, S, N, C = X.shape
    nf = len(fixed)
    dX = np.zeros_like(X)
    dout = np.zeros_like(out)
    dW = np.zeros_like(W)
    dW_r = np.zeros_like(W_r)
    dconv = None if conv is None else [np.zeros_like(w) for w in conv]
    for b in range(B):
        Xs = X[b]
        cf = _coeffs_seq(Xs, W, N, C, k, iters, eps)
        s, r, y, sd = router_scores(Xs, W_r, eps)
        ib = route(s, fixed, k) if idx is None else np.asarray(idx[b], dtype=np.int64)
        w = _routed_weights(s, ib, nf)
        u = tfa_components(out[b], conv)
        G = np.take_along_axis(dXp[b], ib[:, :, None], axis=1)              # [S, k, C]
        Xa = np.take_along_axis(Xs, ib[:, :, None], axis=1)
        hpre, hpost = cf["hpre"], cf["hpost"]
        D = np.einsum("sic,xsc->six", G, u)                                  # <G_i, u_c>
        d_hres = np.einsum("sic,sjc->sij", G, Xa)
        d_hpost = D * w[:, :, None]
        d_w = np.einsum("six,six->si", hpost, D)                             # dL/dw_i
        d_hpre = np.einsum("sc,snc->sn", dx_in[b], Xs) if dx_in is not None else np.zeros((S, N))
        dZ = sinkhorn_reverse(d_hres, cf["trace"])
        dz = np.concatenate([d_hpre * hpre * (1.0 - hpre),
                             (d_hpost * hpost * (1.0 - hpost)).reshape(S, 4 * k),
                             dZ.reshape(S, k * k)], axis=1)
        rstd, p, v = cf["rstd"], cf["p"], cf["v"]
        dp = rstd[:, None] * dz
        drstd = (dz * p).sum(axis=1)
        dv = dp @ W + (drstd * (-(rstd ** 3) / (N * C)))[:, None] * v
        dW += dp.T @ v
        # router: scores of the routed slots scale their write-back
        ds = np.zeros((S, N))
        rows = np.arange(S)
        for i in range(nf, k):
            ds[rows, ib[:, i]] += d_w[:, i]
        dr = ds * s * (1.0 - s)
        dW_r += dr.T @ y
        dy = dr @ W_r
        dv += (dy - dy.mean(axis=1, keepdims=True) - y * (dy * y).mean(axis=1, keepdims=True)) / sd[:, None]
        dXs = dv.reshape(S, N, C).copy()
        if dx_in is not None:
            dXs += hpre[:, :, None] * dx_in[b][:, None, :]
        # per-token sparse write: a stream passes dX' through unless active
        active = np.zeros((S, N), dtype=bool)
        np.put_along_axis(active, ib, True, axis=1)
        dXs += np.where(active[:, :, None], 0.0, dXp[b])
        back = np.einsum("sij,sic->sjc", cf["hres"], G)                      # to X[a_j]
        for j in range(k):
            dXs[rows, ib[:, j]] += back[:, j]
        dX[b] = dXs
        du = np.einsum("six,sic->xsc", hpost * w[:, :, None], G)
        dout_b = du[0].copy()
        if conv is not None:
            for j, wj in enumerate(conv, start=1):
                K = wj.shape[1]
                for tau in range(min(K, S)):
                    dout_b[: S - tau, :] += wj[None, :, tau] * du[j, tau:, :]
                    dconv[j - 1][:, tau] += (du[j, tau:, :] * out[b][: S - tau, :]).sum(axis=0)
        dout[b] = dout_b
    return dict(dX=dX, dout=dout, dconv=dconv, dW=dW, dW_r=dW_r)


def max_rel_err(got, ref):
    """Error measure used by every parity check: max_i |g_i - r_i| /
    max(|r_i|, rms(r)) -- elementwise relative, floored at the tensor's RMS so
    that entries near zero do not dominate."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    floor = np.maximum(np.abs(ref), rms)
    floor = np.where(floor == 0.0, 1.0, floor)
    return float(np.max(np.abs(got - ref) / floor))
