"""CPU oracle for the rank-gated tensor-train (TT) linear layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the library calls this module; only the
tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg do.
It shares no code with the CUDA path.  Everything runs in float64 numpy on
the values it is given (float32 / bf16-representable inputs are exact in
float64), with library matmuls as single steps and no blocking or fusion.

What it computes, following the CoMERA project page (CoMERA: Computing- and
Memory-Efficient Training via Rank-Adaptive Tensor Optimization), section
"Learn the ranks while training" and its rank-control-diagonal figure, and
section "Making small tensor operations fast on GPUs", bullet "One
contraction order for both passes":

* A weight W (M x N, M = prod m_i, N = prod n_j) is a chain of 2d cores
  G_k of shape (r_{k-1}, s_k, r_k), r_0 = r_2d = 1, with the input modes
  first, s = (n_1..n_d, m_1..m_d), and a diagonal D_k on every internal
  link k = 1..2d-1 (the rank of a link is the number of nonzeros of D_k).
  With j = (j_1..j_d) and i = (i_1..i_d) linearised row-major,

      W[i, j] = G_1[0, j_1, :] D_1 G_2[:, j_2, :] D_2 ... D_d ... G_2d[:, i_d, 0]

* The layer computes y[t, i] = sum_j W[i, j] x[t, j]; backward for the
  linear functional L = <dy, y> gives dx = dy W, and dG_k = dL/dG_k,
  dD_k = dL/dD_k.
* A zero entry D_k[a] drops slice a of G_k and G_{k+1}; the layer must then
  equal the rank-truncated TT.  The truncated TT has no parameter D_k[a], so
  the returned gradient dD_k[a] is zero there ("prune convention"); the
  untruncated derivative is also available for finite-difference checks.

Two modes:
  O1 ("dense")   build W explicitly and use y = x W^T, dx = dy W, dW = dy^T x,
                 core and diagonal gradients from full-chain environments.
                 O(T N M): tiny and medium shapes.
  O2 ("chained") the page's contraction order: merge the input-side cores
                 into A (N x r_d) and the output-side cores into B (r_d x M),
                 z = x A, z' = z diag(D_d), y = z' B, and the matching
                 backward.  O(T r (N + M)): used at full workload sizes.

Readings where the pages are silent are listed in the design notes of the
repository: input modes precede output modes, row-major linearisation, a
diagonal on every internal link including the middle one, no bias, GELU in
its exact erf form.
"""

from __future__ import annotations

import itertools
from typing import List, Sequence, Tuple

import numpy as np
from scipy.special import erf

F64 = np.float64


# ---------------------------------------------------------------------------
# shapes


def rank_caps(in_modes: Sequence[int], out_modes: Sequence[int], R: int) -> List[int]:
    """r_k = min(R, prod s_<=k, prod s_>k), r_0 = r_2d = 1.

    Reading of the rank table "Internal tensor-train ranks of each layer in
    one encoder block" (CoMERA project page, "Results"): a requested rank of
    30 appears as 12 or 16 on the end links, which is exactly the product of
    the modes on the short side of the link.
    """
    s = list(in_modes) + list(out_modes)
    K = len(s)
    r = [1]
    for k in range(1, K):
        left = int(np.prod(s[:k]))
        right = int(np.prod(s[k:]))
        r.append(min(R, left, right))
    r.append(1)
    return r


def _modes(cores: Sequence[np.ndarray]) -> List[int]:
    return [c.shape[1] for c in cores]


# ---------------------------------------------------------------------------
# O1: dense reconstruction


def dense_weight_bruteforce(cores, diags, d: int) -> np.ndarray:
    """W[i, j] by summing the definition term by term.  Tiny shapes only.

    Loops over every (j, i) and every assignment of the 2d-1 link indices;
    used to pin :func:`dense_weight`.
    """
    import itertools

    s = _modes(cores)
    K = 2 * d
    ranks = [1] + [c.shape[2] for c in cores]
    N = int(np.prod(s[:d]))
    M = int(np.prod(s[d:]))
    W = np.zeros((M, N), F64)
    for idx in itertools.product(*[range(n) for n in s]):
        jj = 0
        for k in range(d):
            jj = jj * s[k] + idx[k]
        ii = 0
        for k in range(d, K):
            ii = ii * s[k] + idx[k]
        acc = 0.0
        for links in itertools.product(*[range(ranks[k]) for k in range(1, K)]):
            a = (0,) + links + (0,)
            term = 1.0
            for k in range(K):
                term *= float(cores[k][a[k], idx[k], a[k + 1]])
            for k in range(K - 1):
                term *= float(diags[k][a[k + 1]])
            acc += term
        W[ii, jj] = acc
    return W


def chain_product(cores, diags) -> np.ndarray:
    """Contract a chain C_0 E_0 C_1 E_1 ... C_{K-1} into (r_left, prod s, r_right).

    Left to right: the running product P (r_left * S_<k, r_k) is scaled by
    the diagonal on link k, then multiplied with C_k reshaped to
    (r_k, s_k * r_{k+1}).
    """
    K = len(cores)
    c0 = np.asarray(cores[0], F64)
    rl = c0.shape[0]
    P = c0.reshape(rl * c0.shape[1], c0.shape[2])
    for k in range(1, K):
        ck = np.asarray(cores[k], F64)
        P = P * np.asarray(diags[k - 1], F64)[None, :]
        P = P @ ck.reshape(ck.shape[0], ck.shape[1] * ck.shape[2])
        P = P.reshape(-1, ck.shape[2])
    S = int(np.prod(_modes(cores)))
    return P.reshape(rl, S, P.shape[1])


def dense_weight(cores, diags, d: int) -> np.ndarray:
    """W (M x N) from the full chain (input modes first, then output modes)."""
    V = chain_product(cores, diags)          # (1, N*M, 1), index (j, i)
    s = _modes(cores)
    N = int(np.prod(s[:d]))
    M = int(np.prod(s[d:]))
    return V.reshape(N, M).T.copy()


def chain_grads(cores, diags, dOut) -> Tuple[List[np.ndarray], List[np.ndarray]]:
    """Gradients of <dOut, chain_product(cores, diags)> w.r.t. every core and diagonal.

    Out[al, u, s, v, om] = sum L_k[al, u, p] C_k[p, s, q] R_k[q, v, om] where
    L_k = C_0 E_0 ... C_{k-1} E_{k-1} (identity for k = 0) is the left
    environment and R_k = E_k C_{k+1} ... C_{K-1} (identity for the last core)
    the right one.  So dC_k[p, s, q] = sum dOut[al, u, s, v, om] L_k[al, u, p]
    R_k[q, v, om], and dE_k[c] = sum dOut P_k[al, u, c] Q_k[c, v, om] with
    P_k = C_0 .. C_k and Q_k = C_{k+1} .. C_{K-1}.
    """
    K = len(cores)
    s = _modes(cores)
    rl = cores[0].shape[0]
    rr = cores[-1].shape[2]
    dOut = np.asarray(dOut, F64).reshape(rl, int(np.prod(s)), rr)

    def left_env(k):
        # (rl, S_<k, r_k), including the diagonal on link k-1
        if k == 0:
            return np.eye(rl, dtype=F64).reshape(rl, 1, rl)
        P = chain_product(cores[:k], diags[:k - 1])
        return P * np.asarray(diags[k - 1], F64)[None, None, :]

    def right_env(k):
        # (r_{k+1}, S_>k, rr), including the diagonal on link k
        if k == K - 1:
            return np.eye(rr, dtype=F64).reshape(rr, 1, rr)
        Q = chain_product(cores[k + 1:], diags[k + 1:])
        return Q * np.asarray(diags[k], F64)[:, None, None]

    dC = []
    for k in range(K):
        Sl = int(np.prod(s[:k]))
        Sr = int(np.prod(s[k + 1:]))
        G = dOut.reshape(rl, Sl, s[k], Sr, rr)
        L = left_env(k)
        R = right_env(k)
        dC.append(np.einsum("ausvw,aup,qvw->psq", G, L, R, optimize=True))
    dE = []
    for k in range(K - 1):
        Sl = int(np.prod(s[:k + 1]))
        Sr = int(np.prod(s[k + 1:]))
        G = dOut.reshape(rl, Sl, Sr, rr)
        P = chain_product(cores[:k + 1], diags[:k])
        Q = chain_product(cores[k + 1:], diags[k + 1:])
        dE.append(np.einsum("auvw,auc,cvw->c", G, P, Q, optimize=True))
    return dC, dE


def dense_forward(cores, diags, d, x):
    W = dense_weight(cores, diags, d)
    return np.asarray(x, F64) @ W.T


def dense_backward(cores, diags, d, x, dy, prune_convention=True):
    """O1 backward: (dx, dcores, ddiags) from the explicit W."""
    x = np.asarray(x, F64)
    dy = np.asarray(dy, F64)
    W = dense_weight(cores, diags, d)
    dx = dy @ W
    dW = dy.T @ x                                  # (M, N)
    dV = dW.T.reshape(1, -1, 1)                   # index (j, i) as in the chain
    dC, dE = chain_grads(cores, diags, dV)
    if prune_convention:
        dE = [np.where(np.asarray(e) == 0.0, 0.0, g) for e, g in zip(diags, dE)]
    return dx, dC, dE


# ---------------------------------------------------------------------------
# O2: the page's contraction order


def merge_input(cores, diags, d) -> np.ndarray:
    """A (N x r_d) = G_1 D_1 G_2 ... D_{d-1} G_d, without the middle diagonal D_d."""
    P = chain_product(cores[:d], diags[:d - 1])   # (1, N, r_d)
    return P[0]


def merge_output(cores, diags, d) -> np.ndarray:
    """B (r_d x M) = G_{d+1} D_{d+1} ... G_2d."""
    P = chain_product(cores[d:], diags[d:])       # (r_d, M, 1)
    return P[:, :, 0]


def chained_forward(cores, diags, d, x, return_intermediates=False):
    """y = ((x A) diag(D_d)) B.  Returns y, or (y, z) with z = x A."""
    x = np.asarray(x, F64)
    A = merge_input(cores, diags, d)
    B = merge_output(cores, diags, d)
    Dm = np.asarray(diags[d - 1], F64)
    z = x @ A
    y = (z * Dm[None, :]) @ B
    return (y, z) if return_intermediates else y


def chained_backward(cores, diags, d, x, dy, prune_convention=True):
    """O2 backward: dx, dcores, ddiags following the same merge order.

    dz' = dy B^T, dB = z'^T dy, dD_d = sum_t z * dz', dz = dz' diag(D_d),
    dx = dz A^T, dA = x^T dz; then the merges are differentiated with their
    left and right environments (:func:`chain_grads`).
    """
    x = np.asarray(x, F64)
    dy = np.asarray(dy, F64)
    A = merge_input(cores, diags, d)
    B = merge_output(cores, diags, d)
    Dm = np.asarray(diags[d - 1], F64)
    z = x @ A
    zp = z * Dm[None, :]
    dzp = dy @ B.T
    dB = zp.T @ dy
    dDm = np.sum(z * dzp, axis=0)
    dz = dzp * Dm[None, :]
    dx = dz @ A.T
    dA = x.T @ dz
    dCin, dEin = chain_grads(cores[:d], diags[:d - 1], dA.reshape(1, -1, A.shape[1]))
    dCout, dEout = chain_grads(cores[d:], diags[d:], dB.reshape(B.shape[0], -1, 1))
    dC = dCin + dCout
    dE = dEin + [dDm] + dEout
    if prune_convention:
        dE = [np.where(np.asarray(e) == 0.0, 0.0, g) for e, g in zip(diags, dE)]
    return dx, dC, dE


# ---------------------------------------------------------------------------
# rank truncation


def truncate(cores, diags):
    """Delete every slice whose diagonal entry is exactly zero.

    A zero D_k[a] drops slice a (last axis) of G_k and slice a (first axis)
    of G_{k+1}, and the entry itself.  Returns (cores, diags, kept) with
    kept[k] the surviving indices of link k.  A link with no surviving entry
    keeps rank 0, i.e. the layer is removed (it computes zero).
    """
    K = len(cores)
    kept = [np.flatnonzero(np.asarray(e) != 0.0) for e in diags]
    new_cores = []
    for k in range(K):
        c = np.asarray(cores[k])
        if k > 0:
            c = c[kept[k - 1], :, :]
        if k < K - 1:
            c = c[:, :, kept[k]]
        new_cores.append(c)
    new_diags = [np.asarray(e)[kk] for e, kk in zip(diags, kept)]
    return new_cores, new_diags, kept


# ---------------------------------------------------------------------------
# FFN pair with GELU


def gelu(h):
    """Exact GELU: h * Phi(h) = h/2 (1 + erf(h / sqrt 2))."""
    h = np.asarray(h, F64)
    return 0.5 * h * (1.0 + erf(h / np.sqrt(2.0)))


def gelu_grad(h):
    """d/dh GELU = Phi(h) + h phi(h)."""
    h = np.asarray(h, F64)
    Phi = 0.5 * (1.0 + erf(h / np.sqrt(2.0)))
    phi = np.exp(-0.5 * h * h) / np.sqrt(2.0 * np.pi)
    return Phi + h * phi


def ffn_forward(up, down, d_up, d_down, x, return_intermediates=False):
    """y = TT_down(GELU(TT_up(x))).  up/down are (cores, diags) pairs."""
    h = chained_forward(up[0], up[1], d_up, x)
    a = gelu(h)
    y = chained_forward(down[0], down[1], d_down, a)
    return (y, h) if return_intermediates else y


def ffn_backward(up, down, d_up, d_down, x, dy, prune_convention=True):
    """Backward of the FFN pair: dx and (dcores, ddiags) of both layers."""
    h = chained_forward(up[0], up[1], d_up, x)
    a = gelu(h)
    da, dC2, dE2 = chained_backward(down[0], down[1], d_down, a, dy, prune_convention)
    dh = da * gelu_grad(h)
    dx, dC1, dE1 = chained_backward(up[0], up[1], d_up, x, dh, prune_convention)
    return dx, (dC1, dE1), (dC2, dE2)


# ---------------------------------------------------------------------------
# comparison metric


def rel_err(out, ref) -> float:
    """Norm-wise relative error ||out - ref||_F / ||ref||_F (0/0 -> 0, x/0 -> inf)."""
    out = np.asarray(out, F64)
    ref = np.asarray(ref, F64)
    num = float(np.linalg.norm((out - ref).ravel()))
    den = float(np.linalg.norm(ref.ravel()))
    if den == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return num / den


# ---------------------------------------------------------------------------
# Rank-adaptive step (project page, "Learn the ranks while training": the
# early-stage objective  L(G, D) + gamma * S_hat(D) + beta * ||G||^2, where
# S_hat is an l1 penalty on the diagonals standing in for counting their
# nonzeros, and beta ||G||^2 keeps the cores from growing).
#
# Reading (the pages print no formula for S_hat beyond "an l1 penalty on the
# diagonals"): S_hat(D) = sum_k ||D_k||_1 over every internal link, and
# ||G||^2 = sum_k ||G_k||_F^2 over every core.


def penalty(cores, diags, gamma: float, beta: float) -> float:
    """gamma * sum_k |D_k|_1 + beta * sum_k ||G_k||_F^2, in float64."""
    s = sum(float(np.abs(np.asarray(e, F64)).sum()) for e in diags)
    g = sum(float((np.asarray(c, F64) ** 2).sum()) for c in cores)
    return gamma * s + beta * g


def penalty_grads(cores, diags, gamma: float, beta: float):
    """Sub-gradient of `penalty`: 2 beta G_k for the cores and gamma sign(D_k)
    for the diagonals, with sign(0) = 0 (a pruned entry gets no push)."""
    dC = [2.0 * beta * np.asarray(c, F64) for c in cores]
    dE = [gamma * np.sign(np.asarray(e, F64)) for e in diags]
    return dC, dE


def soft_threshold(v, t):
    """Proximal map of t |u|: argmin_u 0.5 (u - v)^2 + t |u|."""
    v = np.asarray(v, F64)
    return np.sign(v) * np.maximum(np.abs(v) - t, 0.0)


def rank_update_f32(cores, diags, dcores, ddiags, gamma: float, beta: float, lr: float):
    """The rank-adaptive step in float32 arithmetic, one rounding per
    operation in the order below (the library applies the same operations
    without contraction, so the two agree bit for bit; the zero / nonzero
    decision of the threshold is a float32 comparison on both sides).

    lr == 0: only the penalty's sub-gradient is added to the gradients,
        dG <- dG + (2 beta) G,   dD <- dD + gamma sign(D).
    lr > 0: one proximal gradient step on the whole objective,
        G <- G - lr (dG + (2 beta) G),
        D <- soft_threshold(D - lr dD, lr gamma),
    so diagonal entries that reach zero are pruned (the next call compacts
    them out).  Returns (cores, diags, dcores, ddiags) as float32 arrays."""
    f = np.float32
    b2 = f(2.0) * f(beta)
    g, lr_, t = f(gamma), f(lr), f(lr) * f(gamma)
    oc, od, odc, odd = [], [], [], []
    for c, dc in zip(cores, dcores):
        c = np.asarray(c, f); dc = np.asarray(dc, f)
        grad = (dc + (b2 * c).astype(f)).astype(f)
        if lr == 0:
            oc.append(c.copy()); odc.append(grad)
        else:
            oc.append((c - (lr_ * grad).astype(f)).astype(f)); odc.append(dc.copy())
    for e, de in zip(diags, ddiags):
        e = np.asarray(e, f); de = np.asarray(de, f)
        if lr == 0:
            sgn = np.where(e > 0, g, np.where(e < 0, -g, f(0.0))).astype(f)
            od.append(e.copy()); odd.append((de + sgn).astype(f))
        else:
            v = (e - (lr_ * de).astype(f)).astype(f)
            out = np.where(v > t, (v - t).astype(f), np.where(v < -t, (v + t).astype(f), f(0.0)))
            od.append(out.astype(f)); odd.append(de.copy())
    return oc, od, odc, odd


# ---------------------------------------------------------------------------
# TT-matrix (TTM) embedding table (project page: "Embedding tables, whose
# shapes are very unbalanced, use the related tensor-train-matrix format";
# poster digest, TT/TTM figure: each core F_k carries an index pair
# (m_k, n_k)).  E (V x Dm), V = prod m_k, Dm = prod n_k, row index
# i = (i_1..i_d) and column index j = (j_1..j_d) row-major:
#
#     E[i, j] = F_1[0, i_1, j_1, :] D_1 F_2[:, i_2, j_2, :] D_2 ... F_d[:, i_d, j_d, 0]
#
# A lookup returns the rows E[idx[b], :]; its backward, for the functional
# L = <dout, rows>, gives every dF_k and dD_k (duplicated indices add up).


def _row_digits(rows, row_modes):
    rows = np.asarray(rows, np.int64)
    dig = []
    rem = rows.copy()
    for m in reversed(row_modes):
        dig.append(rem % m)
        rem //= m
    return list(reversed(dig))


def ttm_table_bruteforce(cores, diags) -> np.ndarray:
    """The whole table by the explicit sum over every rank index (tiny shapes)."""
    d = len(cores)
    m = [c.shape[1] for c in cores]
    n = [c.shape[2] for c in cores]
    V, Dm = int(np.prod(m)), int(np.prod(n))
    E = np.zeros((V, Dm), F64)
    ranges = [range(c.shape[3]) for c in cores[:-1]]
    for i in range(V):
        ii = np.unravel_index(i, m)
        for j in range(Dm):
            jj = np.unravel_index(j, n)
            s = 0.0
            for a in itertools.product(*ranges):
                p = 1.0
                prev = 0
                for k in range(d):
                    nxt = a[k] if k < d - 1 else 0
                    p *= float(cores[k][prev, ii[k], jj[k], nxt])
                    if k < d - 1:
                        p *= float(diags[k][a[k]])
                    prev = nxt
                s += p
            E[i, j] = s
    return E


def _ttm_prefix(cores, diags, dig, k_end):
    """P (U, n_1..n_k flattened, r_k): the chain through cores 0..k_end-1,
    with the diagonals between them but not the one after core k_end-1."""
    U = dig[0].shape[0]
    P = np.ones((U, 1, 1), F64)
    for k in range(k_end):
        if k > 0:
            P = P * np.asarray(diags[k - 1], F64)[None, None, :]
        Fk = np.asarray(cores[k], F64)[:, dig[k], :, :].transpose(1, 0, 2, 3)  # (U, r, n, r')
        P = np.einsum("ulb,ubjc->uljc", P, Fk).reshape(U, -1, Fk.shape[3])
    return P


def _ttm_suffix(cores, diags, dig, k_begin):
    """S (U, r_{k_begin}, n_{k_begin+1}..n_d flattened): the chain through
    cores k_begin..d-1 (0-based), with the diagonals between them but not the
    one before core k_begin."""
    d = len(cores)
    U = dig[0].shape[0]
    S = np.ones((U, 1, 1), F64)
    for k in range(d - 1, k_begin - 1, -1):
        if k < d - 1:
            S = np.asarray(diags[k], F64)[None, :, None] * S
        Fk = np.asarray(cores[k], F64)[:, dig[k], :, :].transpose(1, 0, 2, 3)  # (U, r, n, r')
        S = np.einsum("ubjc,ucr->ubjr", Fk, S).reshape(U, Fk.shape[1], -1)
    return S


def ttm_rows(cores, diags, rows) -> np.ndarray:
    """Rows E[rows, :] by the chained contraction (float64)."""
    m = [c.shape[1] for c in cores]
    dig = _row_digits(rows, m)
    P = _ttm_prefix(cores, diags, dig, len(cores))
    return P[:, :, 0].copy()


def ttm_lookup(cores, diags, idx) -> np.ndarray:
    """out[b] = E[idx[b]]: each distinct row is computed once."""
    uniq, inv = np.unique(np.asarray(idx, np.int64), return_inverse=True)
    return ttm_rows(cores, diags, uniq)[inv]


def ttm_lookup_backward(cores, diags, idx, dout, prune_convention=True):
    """dF_k and dD_k of L = <dout, ttm_lookup(idx)>: gradients of repeated
    indices are summed first (one gradient row per distinct index)."""
    d = len(cores)
    m = [c.shape[1] for c in cores]
    uniq, inv = np.unique(np.asarray(idx, np.int64), return_inverse=True)
    dR = np.zeros((uniq.size, np.asarray(dout).shape[1]), F64)
    np.add.at(dR, inv, np.asarray(dout, F64))
    dig = _row_digits(uniq, m)
    U = uniq.size
    dC = [np.zeros_like(np.asarray(c, F64)) for c in cores]
    dE = [np.zeros(np.asarray(e).shape, F64) for e in diags]
    for k in range(d):
        Pl = _ttm_prefix(cores, diags, dig, k)          # (U, left, r_{k-1}) without D_{k-1}
        if k > 0:
            Pl = Pl * np.asarray(diags[k - 1], F64)[None, None, :]
        Sr = _ttm_suffix(cores, diags, dig, k + 1)      # (U, r_k, right) without D_k
        if k < d - 1:
            Sr = np.asarray(diags[k], F64)[None, :, None] * Sr
        nk = cores[k].shape[2]
        G = dR.reshape(U, Pl.shape[1], nk, Sr.shape[2])
        contrib = np.einsum("ulb,uljr,ucr->ubjc", Pl, G, Sr)   # (U, r_{k-1}, n_k, r_k)
        acc = np.zeros((cores[k].shape[1],) + contrib.shape[1:], F64)
        np.add.at(acc, dig[k], contrib)
        dC[k] = acc.transpose(1, 0, 2, 3).copy()
    for k in range(d - 1):
        P = _ttm_prefix(cores, diags, dig, k + 1)      # through core k, no D_k
        S = _ttm_suffix(cores, diags, dig, k + 1)      # from core k+1, no D_k
        G = dR.reshape(U, P.shape[1], S.shape[2])
        g = np.einsum("ulc,ulr,ucr->c", P, G, S)
        if prune_convention:
            g = np.where(np.asarray(diags[k]) == 0, 0.0, g)
        dE[k] = g
    return dC, dE
