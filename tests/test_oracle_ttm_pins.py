"""Pins for the oracle's TT-matrix (TTM) embedding lookup.

Each test ties the oracle to something it cannot agree with by construction:
the explicit sum of the definition, the Kronecker closed form at rank 1,
Oseledets' TT-SVD of a random table with paired (row, column) mode indices,
central finite differences, and exact identities (repeated indices,
homogeneity).
"""

import numpy as np
import pytest

from oracle import tt_oracle as O
from tensor_train_compressed_tt_gb300 import synth


def _random_ttm(rng, m, n, r, diag_lo=0.5):
    cores = [rng.standard_normal((r[k], m[k], n[k], r[k + 1])) for k in range(len(m))]
    diags = [rng.uniform(diag_lo, 1.5, r[k]) for k in range(1, len(m))]
    return cores, diags


SHAPES = [((2, 3), (2, 2), (1, 3, 1)),
          ((2, 3, 2), (2, 2, 3), (1, 2, 3, 1)),
          ((3, 1, 2), (1, 2, 2), (1, 2, 2, 1))]


@pytest.mark.parametrize("m,n,r", SHAPES)
def test_chain_equals_bruteforce_sum(m, n, r):
    rng = np.random.Generator(np.random.PCG64(31))
    cores, diags = _random_ttm(rng, m, n, r)
    E = O.ttm_table_bruteforce(cores, diags)
    V = int(np.prod(m))
    np.testing.assert_allclose(O.ttm_rows(cores, diags, np.arange(V)), E, rtol=1e-12, atol=1e-12)


def test_rank_one_is_a_kronecker_product():
    rng = np.random.Generator(np.random.PCG64(32))
    m, n, r = (2, 3, 2), (3, 2, 2), (1, 1, 1, 1)
    cores, diags = _random_ttm(rng, m, n, r)
    K = cores[0][0, :, :, 0]
    for k in range(1, 3):
        K = np.kron(K, cores[k][0, :, :, 0])
    K = K * diags[0][0] * diags[1][0]
    np.testing.assert_allclose(O.ttm_rows(cores, diags, np.arange(12)), K, rtol=1e-12)


def _ttm_svd(E, m, n):
    """Oseledets' TT-SVD of E reshaped with paired (m_k, n_k) modes."""
    d = len(m)
    T = E.reshape(tuple(m) + tuple(n))
    T = T.transpose([x for k in range(d) for x in (k, d + k)])  # (m1, n1, m2, n2, ...)
    C = T.reshape(-1)
    cores, diags = [], []
    r = 1
    for k in range(d - 1):
        C = C.reshape(r * m[k] * n[k], -1)
        U, S, Vt = np.linalg.svd(C, full_matrices=False)
        cores.append(U.reshape(r, m[k], n[k], S.size))
        diags.append(S)
        C = Vt
        r = S.size
    cores.append(C.reshape(r, m[-1], n[-1], 1))
    return cores, diags


@pytest.mark.parametrize("m,n", [((2, 3), (3, 2)), ((2, 2, 3), (2, 3, 1))])
def test_ttm_svd_reconstructs_random_table(m, n):
    rng = np.random.Generator(np.random.PCG64(33))
    V, Dm = int(np.prod(m)), int(np.prod(n))
    E = rng.standard_normal((V, Dm))
    cores, diags = _ttm_svd(E, m, n)
    np.testing.assert_allclose(O.ttm_rows(cores, diags, np.arange(V)), E, rtol=1e-11, atol=1e-11)
    idx = rng.integers(0, V, 9)
    np.testing.assert_allclose(O.ttm_lookup(cores, diags, idx), E[idx], rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("m,n,r", SHAPES)
def test_lookup_gradients_match_finite_differences(m, n, r):
    rng = np.random.Generator(np.random.PCG64(34))
    cores, diags = _random_ttm(rng, m, n, r)
    V, Dm = int(np.prod(m)), int(np.prod(n))
    idx = np.array([1, V - 1, 1, 0, V - 1, 1])   # repeated indices
    dout = rng.standard_normal((idx.size, Dm))
    dC, dE = O.ttm_lookup_backward(cores, diags, idx, dout, prune_convention=False)
    L = lambda c, e: float(np.sum(dout * O.ttm_lookup(c, e, idx)))
    h = 1e-6
    for k, c in enumerate(cores):
        for pos in np.ndindex(*c.shape):
            cp = [x.copy() for x in cores]; cm = [x.copy() for x in cores]
            cp[k][pos] += h; cm[k][pos] -= h
            fd = (L(cp, diags) - L(cm, diags)) / (2 * h)
            assert abs(fd - dC[k][pos]) <= 1e-6 * max(1.0, abs(fd))
    for k, e in enumerate(diags):
        for a in range(e.size):
            ep = [x.copy() for x in diags]; em = [x.copy() for x in diags]
            ep[k][a] += h; em[k][a] -= h
            fd = (L(cores, ep) - L(cores, em)) / (2 * h)
            assert abs(fd - dE[k][a]) <= 1e-6 * max(1.0, abs(fd))


def test_repeated_indices_add_their_gradients():
    """Looking a row up twice with gradients g1, g2 equals looking it up once
    with g1 + g2; the forward rows are copies."""
    rng = np.random.Generator(np.random.PCG64(35))
    m, n, r = (2, 3, 2), (2, 2, 3), (1, 2, 3, 1)
    cores, diags = _random_ttm(rng, m, n, r)
    idx = np.array([4, 7, 4, 4, 9])
    dout = rng.standard_normal((5, 12))
    out = O.ttm_lookup(cores, diags, idx)
    assert np.array_equal(out[0], out[2]) and np.array_equal(out[0], out[3])
    a = O.ttm_lookup_backward(cores, diags, idx, dout)
    b = O.ttm_lookup_backward(cores, diags, np.array([4, 7, 9]),
                              np.stack([dout[0] + dout[2] + dout[3], dout[1], dout[4]]))
    for x, y in zip(a[0] + a[1], b[0] + b[1]):
        np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-12)


def test_homogeneity_and_prune_convention():
    """L is linear in each core and each diagonal: <F_k, dF_k> = <D_k, dD_k> = L.
    A zero diagonal entry gets dD = 0 (the truncated table has no such entry)."""
    rng = np.random.Generator(np.random.PCG64(36))
    m, n, r = (3, 2, 2), (2, 3, 2), (1, 3, 2, 1)
    cores, diags = _random_ttm(rng, m, n, r)
    idx = rng.integers(0, 12, 20)
    dout = rng.standard_normal((20, 12))
    L = float(np.sum(dout * O.ttm_lookup(cores, diags, idx)))
    dC, dE = O.ttm_lookup_backward(cores, diags, idx, dout)
    for c, g in zip(cores, dC):
        assert abs(float(np.sum(c * g)) - L) <= 1e-10 * max(1.0, abs(L))
    for e, g in zip(diags, dE):
        assert abs(float(np.sum(e * g)) - L) <= 1e-10 * max(1.0, abs(L))
    diags[0][1] = 0.0
    _, dE0 = O.ttm_lookup_backward(cores, diags, idx, dout)
    assert dE0[0][1] == 0.0


def test_zipf_indices_repeat_and_stay_in_range():
    w = synth.TTM_WORKLOADS["ttm_emb_10k"]
    t = synth.draw_ttm(w)
    assert t.idx.dtype == np.int32 and t.idx.min() >= 0 and t.idx.max() < w.vocab
    assert np.unique(t.idx).size < t.idx.size // 2   # many repeated rows
