"""Pins for the CPU oracle against facts fixed outside the oracle itself.

Each test ties the oracle to something it cannot agree with by construction:
a brute-force sum of the definition, a closed form (Kronecker products), a
library decomposition (SVD / TT-SVD), the printed rank table, finite
differences, or an exact identity of the mathematics (homogeneity, gauge).
"""

import os

import numpy as np
import pytest
from scipy.stats import norm

from oracle import tt_oracle as O
from tensor_train_compressed_tt_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _random_tt(rng, shape, diag="uniform"):
    li = synth.draw_layer(rng, shape, 0.7, diag)
    return [c.astype(np.float64) for c in li.cores], [e.astype(np.float64) for e in li.diags]


SMALL_SHAPES = [
    synth.LayerShape((2,), (3,), (1, 2, 1)),
    synth.LayerShape((2, 3), (3, 2), (1, 2, 3, 2, 1)),
    synth.LayerShape((3, 2), (2, 2), (1, 3, 2, 2, 1)),
    synth.LayerShape((2, 1, 2), (2, 2, 1), (1, 2, 2, 3, 2, 1, 1)),
]


# --- rank plan --------------------------------------------------------------


def _read_rank_table():
    rows = []
    with open(os.path.join(GOLDEN, "rank_table.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            name, im, om, R, rk = line.split()
            rows.append((name, [int(v) for v in im.split(",")], [int(v) for v in om.split(",")],
                         int(R), [int(v) for v in rk.split(",")]))
    return rows


def test_rank_caps_reproduce_printed_table():
    rows = _read_rank_table()
    assert len(rows) == 6
    for name, im, om, R, printed in rows:
        r = O.rank_caps(im, om, R)
        assert r[0] == 1 and r[-1] == 1
        assert r[1:-1] == printed, name


def test_workload_ranks_are_capped_ranks():
    for w in synth.WORKLOADS.values():
        for L in w.layers:
            R = max(L.ranks)
            assert list(L.ranks) == O.rank_caps(L.in_modes, L.out_modes, R), w.name


# --- dense reconstruction -----------------------------------------------------


@pytest.mark.parametrize("shape", SMALL_SHAPES)
def test_dense_weight_equals_bruteforce_definition(rng, shape):
    cores, diags = _random_tt(rng, shape)
    W = O.dense_weight(cores, diags, shape.d)
    Wb = O.dense_weight_bruteforce(cores, diags, shape.d)
    assert W.shape == (shape.M, shape.N)
    np.testing.assert_allclose(W, Wb, rtol=1e-12, atol=1e-13)


def test_rank_one_is_kronecker_product(rng):
    # all ranks 1: W^T, as a vector over (j_1..j_d, i_1..i_d), is the Kronecker
    # product of the per-core vectors times the product of the diagonals
    shape = synth.LayerShape((2, 3, 2), (3, 1, 2), (1, 1, 1, 1, 1, 1, 1))
    cores, diags = _random_tt(rng, shape)
    v = np.array([1.0])
    for c in cores:
        v = np.kron(v, c[0, :, 0])
    v = v * np.prod([e[0] for e in diags])
    Wk = v.reshape(shape.N, shape.M).T
    np.testing.assert_allclose(O.dense_weight(cores, diags, shape.d), Wk, rtol=1e-13, atol=0)
    x = rng.standard_normal((5, shape.N))
    np.testing.assert_allclose(O.chained_forward(cores, diags, shape.d, x), x @ Wk.T,
                               rtol=1e-12, atol=1e-14)


def test_order_one_is_svd(rng):
    # d = 1: W = U diag(S) V^T is a TT with G_1[0] = V, D_1 = S, G_2[:, :, 0] = U^T
    M, N = 7, 5
    W0 = rng.standard_normal((M, N))
    U, S, Vt = np.linalg.svd(W0, full_matrices=False)
    r = S.size
    cores = [Vt.T.reshape(1, N, r), U.T.reshape(r, M, 1)]
    diags = [S]
    np.testing.assert_allclose(O.dense_weight(cores, diags, 1), W0, rtol=1e-12, atol=1e-12)
    x = rng.standard_normal((3, N))
    np.testing.assert_allclose(O.chained_forward(cores, diags, 1, x), x @ W0.T,
                               rtol=1e-12, atol=1e-12)


def _tt_svd(W0, in_modes, out_modes):
    """Oseledets' TT-SVD without truncation; singular values go into the diagonals."""
    s = list(in_modes) + list(out_modes)
    N = int(np.prod(in_modes))
    M = int(np.prod(out_modes))
    C = W0.T.reshape(N * M)               # index (j, i), row-major
    cores, diags = [], []
    r = 1
    for k in range(len(s) - 1):
        C = C.reshape(r * s[k], -1)
        U, S, Vt = np.linalg.svd(C, full_matrices=False)
        rk = S.size
        cores.append(U.reshape(r, s[k], rk))
        diags.append(S)
        C = Vt
        r = rk
    cores.append(C.reshape(r, s[-1], 1))
    return cores, diags


@pytest.mark.parametrize("modes", [((2, 3), (3, 2)), ((2, 2, 2), (3, 1, 2)), ((3,), (4,))])
def test_tt_svd_reconstructs_random_matrix(rng, modes):
    im, om = modes
    N, M = int(np.prod(im)), int(np.prod(om))
    W0 = rng.standard_normal((M, N))
    cores, diags = _tt_svd(W0, im, om)
    d = len(im)
    np.testing.assert_allclose(O.dense_weight(cores, diags, d), W0, rtol=1e-11, atol=1e-11)
    x = rng.standard_normal((4, N))
    np.testing.assert_allclose(O.chained_forward(cores, diags, d, x), x @ W0.T,
                               rtol=1e-11, atol=1e-11)
    dy = rng.standard_normal((4, M))
    dx, _, _ = O.chained_backward(cores, diags, d, x, dy)
    np.testing.assert_allclose(dx, dy @ W0, rtol=1e-11, atol=1e-11)


# --- O1 == O2 -------------------------------------------------------------------


@pytest.mark.parametrize("d", [1, 2, 3, 4])
def test_dense_and_chained_agree(rng, d):
    for _ in range(3):
        shape = synth.random_shape(rng, d, max_mode=3, max_rank=3)
        cores, diags = _random_tt(rng, shape)
        x = rng.standard_normal((5, shape.N))
        dy = rng.standard_normal((5, shape.M))
        y1 = O.dense_forward(cores, diags, d, x)
        y2 = O.chained_forward(cores, diags, d, x)
        assert O.rel_err(y2, y1) < 1e-12
        dx1, dC1, dE1 = O.dense_backward(cores, diags, d, x, dy, prune_convention=False)
        dx2, dC2, dE2 = O.chained_backward(cores, diags, d, x, dy, prune_convention=False)
        assert O.rel_err(dx2, dx1) < 1e-12
        for a, b in zip(dC2, dC1):
            assert O.rel_err(a, b) < 1e-12
        for a, b in zip(dE2, dE1):
            assert O.rel_err(a, b) < 1e-12


# --- truncation -------------------------------------------------------------------


@pytest.mark.parametrize("d", [1, 2, 3])
def test_zeroed_diagonal_equals_truncated_tt(rng, d):
    shape = synth.random_shape(rng, d, max_mode=3, max_rank=4)
    cores, diags = _random_tt(rng, shape)
    # zero at least one entry on every link that has more than one
    for e in diags:
        if e.size > 1:
            e[rng.permutation(e.size)[: e.size // 2]] = 0.0
    tc, td, kept = O.truncate(cores, diags)
    # the truncation really removed the zeroed slices: every link keeps
    # exactly nnz(D_k) ranks, and at least one link lost some
    for k, e in enumerate(diags):
        assert len(kept[k]) == np.count_nonzero(e) == td[k].size
        assert tc[k].shape[2] == tc[k + 1].shape[0] == np.count_nonzero(e)
    assert sum(len(kk) for kk in kept) < sum(e.size for e in diags)
    x = rng.standard_normal((4, shape.N))
    dy = rng.standard_normal((4, shape.M))
    y = O.chained_forward(cores, diags, d, x)
    yt = O.chained_forward(tc, td, d, x)
    assert O.rel_err(y, yt) < 1e-12
    dx, dC, dE = O.chained_backward(cores, diags, d, x, dy)
    dxt, dCt, dEt = O.chained_backward(tc, td, d, x, dy)
    assert O.rel_err(dx, dxt) < 1e-12
    K = 2 * d
    for k in range(K):
        g = dC[k]
        sub = g
        if k > 0:
            sub = sub[kept[k - 1], :, :]
        if k < K - 1:
            sub = sub[:, :, kept[k]]
        assert O.rel_err(sub, dCt[k]) < 1e-12
        # slices that touch a dropped entry have exactly zero gradient
        mask = np.zeros(g.shape, bool)
        if k > 0:
            drop_l = np.setdiff1d(np.arange(g.shape[0]), kept[k - 1])
            mask[drop_l, :, :] = True
        if k < K - 1:
            drop_r = np.setdiff1d(np.arange(g.shape[2]), kept[k])
            mask[:, :, drop_r] = True
        assert np.all(g[mask] == 0.0)
    for k in range(K - 1):
        assert np.all(dE[k][diags[k] == 0.0] == 0.0)
        assert O.rel_err(dE[k][kept[k]], dEt[k]) < 1e-12


def test_truncate_hand_built_example():
    """A hand-built order-2 chain (d = 1: cores (1,2,3), (3,2,1)) with D_1 =
    (2, 0, -1): the truncation keeps ranks 0 and 2 only, i.e. columns 0 and 2
    of G_1's last axis, rows 0 and 2 of G_2's first axis, and D_1 = (2, -1)."""
    G1 = np.arange(6, dtype=np.float64).reshape(1, 2, 3) + 1.0      # values 1..6
    G2 = np.arange(6, dtype=np.float64).reshape(3, 2, 1) + 10.0     # values 10..15
    D1 = np.array([2.0, 0.0, -1.0])
    tc, td, kept = O.truncate([G1, G2], [D1])
    assert kept[0].tolist() == [0, 2]
    assert td[0].tolist() == [2.0, -1.0]
    assert tc[0].shape == (1, 2, 2) and tc[1].shape == (2, 2, 1)
    # G1[0, s, :] = (1,2,3) / (4,5,6) -> keep columns 0 and 2
    assert tc[0][0].tolist() == [[1.0, 3.0], [4.0, 6.0]]
    # G2[:, s, 0] rows 0 and 2: (10, 11) and (14, 15)
    assert tc[1][:, :, 0].tolist() == [[10.0, 11.0], [14.0, 15.0]]
    # the layer itself: W[i, j] = sum_a G1[0,j,a] D1[a] G2[a,i,0], written out
    W = np.array([[sum(G1[0, j, a] * D1[a] * G2[a, i, 0] for a in range(3)) for j in range(2)]
                  for i in range(2)])
    assert np.array_equal(O.dense_weight(tc, td, 1), W)
    # an all-zero link truncates to rank 0 on that link
    tz, dz, kz = O.truncate([G1, G2], [np.zeros(3)])
    assert kz[0].size == 0 and tz[0].shape == (1, 2, 0) and tz[1].shape == (0, 2, 1)


def test_rel_err_hand_values():
    """The comparison metric every parity test uses: ||out - ref|| / ||ref||
    (Frobenius, over all elements), checked on values computed by hand."""
    # difference (0, 1) against a reference of norm sqrt 2
    assert O.rel_err([1.0, 2.0], [1.0, 1.0]) == pytest.approx(1.0 / np.sqrt(2.0), rel=1e-15)
    # divides by the reference's norm, not the output's: |2 - 1| / |1| = 1 (not 1/2)
    assert O.rel_err([2.0, 0.0], [1.0, 0.0]) == 1.0
    # the difference, not the sum: equal tensors give exactly 0
    assert O.rel_err([1.0, -3.0], [1.0, -3.0]) == 0.0
    # a 2-norm over all elements, not a max: (1,1,1,1) vs (0,0,0,2) -> 2 / 2
    assert O.rel_err([1.0, 1.0, 1.0, 1.0], [0.0, 0.0, 0.0, 2.0]) == 1.0
    # every element of a 3-D tensor counts: one 3-4-5 difference in 24 entries
    ref = np.zeros((2, 3, 4))
    ref[1, 2, 3] = 5.0
    out = ref.copy()
    out[0, 0, 0] = 3.0
    out[1, 1, 1] = 4.0
    assert O.rel_err(out, ref) == 1.0
    # zero reference: 0 for a zero output, infinity otherwise
    assert O.rel_err([0.0, 0.0], [0.0, 0.0]) == 0.0
    assert O.rel_err([0.0, 1e-30], [0.0, 0.0]) == float("inf")


def test_all_zero_link_removes_layer(rng):
    shape = synth.LayerShape((2, 3), (3, 2), (1, 2, 3, 2, 1))
    cores, diags = _random_tt(rng, shape)
    diags[1][:] = 0.0
    x = rng.standard_normal((3, shape.N))
    dy = rng.standard_normal((3, shape.M))
    assert np.all(O.chained_forward(cores, diags, 2, x) == 0.0)
    dx, dC, dE = O.chained_backward(cores, diags, 2, x, dy)
    assert np.all(dx == 0.0)
    assert all(np.all(g == 0.0) for g in dC)
    assert all(np.all(g == 0.0) for g in dE)


# --- finite differences -------------------------------------------------------------


def _loss(cores, diags, d, x, dy):
    return float(np.sum(O.chained_forward(cores, diags, d, x) * dy))


@pytest.mark.parametrize("shape", SMALL_SHAPES)
def test_gradients_match_central_differences(rng, shape):
    d = shape.d
    cores, diags = _random_tt(rng, shape)
    x = rng.standard_normal((3, shape.N))
    dy = rng.standard_normal((3, shape.M))
    dx, dC, dE = O.chained_backward(cores, diags, d, x, dy, prune_convention=False)
    h = 1e-6

    def fd(arr, setter):
        g = np.zeros(arr.shape)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + h
            lp = setter()
            arr[idx] = old - h
            lm = setter()
            arr[idx] = old
            g[idx] = (lp - lm) / (2 * h)
        return g

    L = lambda: _loss(cores, diags, d, x, dy)
    assert O.rel_err(dx, fd(x, L)) < 1e-6
    for k in range(2 * d):
        assert O.rel_err(dC[k], fd(cores[k], L)) < 1e-6, k
    for k in range(2 * d - 1):
        assert O.rel_err(dE[k], fd(diags[k], L)) < 1e-6, k


def test_ffn_gradients_match_central_differences(rng):
    up_s = synth.LayerShape((2, 2), (3, 2), (1, 2, 2, 2, 1))
    dn_s = synth.LayerShape((2, 3), (2, 2), (1, 2, 2, 2, 1))
    up = _random_tt(rng, up_s)
    dn = _random_tt(rng, dn_s)
    x = rng.standard_normal((3, up_s.N))
    dy = rng.standard_normal((3, dn_s.M))
    dx, (dC1, dE1), (dC2, dE2) = O.ffn_backward(up, dn, 2, 2, x, dy, prune_convention=False)
    h = 1e-6

    def L():
        return float(np.sum(O.ffn_forward(up, dn, 2, 2, x) * dy))

    def fd(arr):
        g = np.zeros(arr.shape)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + h
            lp = L()
            arr[idx] = old - h
            lm = L()
            arr[idx] = old
            g[idx] = (lp - lm) / (2 * h)
        return g

    assert O.rel_err(dx, fd(x)) < 1e-6
    for k in range(4):
        assert O.rel_err(dC1[k], fd(up[0][k])) < 1e-6
        assert O.rel_err(dC2[k], fd(dn[0][k])) < 1e-6
    for k in range(3):
        assert O.rel_err(dE1[k], fd(up[1][k])) < 1e-6
        assert O.rel_err(dE2[k], fd(dn[1][k])) < 1e-6


# --- GELU -------------------------------------------------------------------------


def test_gelu_against_normal_cdf():
    h = np.linspace(-6, 6, 241)
    np.testing.assert_allclose(O.gelu(h), h * norm.cdf(h), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(O.gelu_grad(h), norm.cdf(h) + h * norm.pdf(h),
                               rtol=1e-12, atol=1e-15)
    assert O.gelu(0.0) == 0.0 and O.gelu_grad(0.0) == 0.5
    eps = 1e-6
    fd = (O.gelu(h + eps) - O.gelu(h - eps)) / (2 * eps)
    np.testing.assert_allclose(O.gelu_grad(h), fd, rtol=1e-7, atol=1e-9)


# --- identities at workload shapes ----------------------------------------------------


@pytest.mark.parametrize("name", ["tiny64_f32", "tt768_bf16", "pruned768_3072_bf16"])
def test_homogeneity_and_gauge(name):
    w = synth.WORKLOADS[name]
    inp = synth.draw(w, seed=0, tokens=64)
    L0 = inp.layers[0]
    d = w.layers[0].d
    cores = [c.astype(np.float64) for c in L0.cores]
    diags = [e.astype(np.float64) for e in L0.diags]
    y = O.chained_forward(cores, diags, d, inp.x)
    dx, dC, dE = O.chained_backward(cores, diags, d, inp.x, inp.dy, prune_convention=True)
    ref = float(np.sum(y * inp.dy))
    # L is linear in x, in every G_k and in every D_k (zeroed entries have zero
    # gradient but contribute D_k[a] dD_k[a] = 0 either way)
    assert abs(float(np.sum(inp.x * dx)) - ref) <= 1e-10 * (abs(ref) + 1)
    for k in range(2 * d):
        assert abs(float(np.sum(cores[k] * dC[k])) - ref) <= 1e-10 * (abs(ref) + 1)
    for k in range(2 * d - 1):
        assert abs(float(np.sum(diags[k] * dE[k])) - ref) <= 1e-10 * (abs(ref) + 1)
    # gauge: scale slice a of link k by c on the left core and 1/c on the right
    k, a, c = 1, 1, 3.0
    g2 = [g.copy() for g in cores]
    g2[k][:, :, a] *= c
    g2[k + 1][a, :, :] /= c
    assert O.rel_err(O.chained_forward(g2, diags, d, inp.x), y) < 1e-12


def test_pack_unpack_roundtrip(rng):
    shape = SMALL_SHAPES[2]
    li = synth.draw_layer(rng, shape, 1.0, "uniform")
    flat = synth.pack(li.cores, li.diags)
    n = sum(int(np.prod(s)) for s in shape.core_shapes()) + sum(shape.diag_sizes())
    assert flat.size == n
    c2, d2 = synth.unpack(shape, flat)
    for a, b in zip(c2, li.cores):
        assert np.array_equal(a, b)
    for a, b in zip(d2, li.diags):
        assert np.array_equal(a, b)


def test_pruned_workload_has_half_zeros():
    w = synth.WORKLOADS["pruned768_3072_bf16"]
    inp = synth.draw(w, seed=0, tokens=8)
    for e in inp.layers[0].diags:
        assert int(np.sum(e == 0.0)) == e.size // 2
        nz = e[e != 0.0]
        assert np.all((nz >= 0.5) & (nz <= 1.5))


def test_bf16_rounding_is_round_to_nearest_even():
    import torch
    v = np.array([1.0, 1.00390625, 1.005859375, -2.5e-3, 3.0e5, 1e-30], np.float32)
    v = np.concatenate([v, np.random.default_rng(0).standard_normal(1000).astype(np.float32)])
    ours = synth.round_bf16(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(ours, ref)


# --- rank-adaptive step (early-stage objective) --------------------------------


def test_penalty_gradient_matches_finite_differences():
    """2 beta G and gamma sign(D) against central differences of the penalty
    value (diagonal entries kept away from the kink at 0)."""
    rng = np.random.Generator(np.random.PCG64(11))
    shape = synth.LayerShape((2, 3), (3, 2), (1, 2, 3, 2, 1))
    cores, diags = _random_tt(rng, shape)
    gamma, beta, h = 0.3, 0.7, 1e-6
    dC, dE = O.penalty_grads(cores, diags, gamma, beta)
    for k, c in enumerate(cores):
        for idx in [(0, 0, 0), tuple(s - 1 for s in c.shape)]:
            cp = [x.copy() for x in cores]; cm = [x.copy() for x in cores]
            cp[k][idx] += h; cm[k][idx] -= h
            fd = (O.penalty(cp, diags, gamma, beta) - O.penalty(cm, diags, gamma, beta)) / (2 * h)
            assert abs(fd - dC[k][idx]) <= 1e-6 * max(1.0, abs(fd))
    for k, e in enumerate(diags):
        for a in range(e.shape[0]):
            ep = [x.copy() for x in diags]; em = [x.copy() for x in diags]
            ep[k][a] += h; em[k][a] -= h
            fd = (O.penalty(cores, ep, gamma, beta) - O.penalty(cores, em, gamma, beta)) / (2 * h)
            assert abs(fd - dE[k][a]) <= 1e-6


def test_soft_threshold_is_the_proximal_map():
    """soft_threshold(v, t) minimises 0.5 (u - v)^2 + t |u| (brute force)."""
    u = np.linspace(-4.0, 4.0, 160001)
    for v in [-2.5, -0.6, -0.2, 0.0, 0.15, 0.9, 3.1]:
        for t in [0.0, 0.25, 1.0]:
            best = u[np.argmin(0.5 * (u - v) ** 2 + t * np.abs(u))]
            assert abs(O.soft_threshold(v, t) - best) <= 1e-4


def test_rank_update_f32_against_float64():
    """The float32 step equals the float64 formulas within float32 rounding,
    and the entries it prunes are exactly those with |D - lr dD| < lr gamma."""
    rng = np.random.Generator(np.random.PCG64(12))
    shape = synth.LayerShape((3, 2), (2, 3), (1, 3, 2, 3, 1))
    cores, diags = _random_tt(rng, shape)
    cores = [c.astype(np.float32).astype(np.float64) for c in cores]
    diags = [e.astype(np.float32).astype(np.float64) for e in diags]
    dC = [rng.standard_normal(c.shape).astype(np.float32).astype(np.float64) for c in cores]
    dE = [rng.standard_normal(e.shape).astype(np.float32).astype(np.float64) for e in diags]
    gamma, beta = 0.5, 0.25
    # gradient-only form
    _, _, gc, ge = O.rank_update_f32(cores, diags, dC, dE, gamma, beta, 0.0)
    pc, pe = O.penalty_grads(cores, diags, gamma, beta)
    for a, b, c in zip(gc, dC, pc):
        np.testing.assert_allclose(a, b + c, rtol=2e-6, atol=1e-6)
    for a, b, c in zip(ge, dE, pe):
        np.testing.assert_allclose(a, b + c, rtol=2e-6, atol=1e-6)
    # proximal step (threshold lr * gamma = 0.8 prunes some entries)
    lr, gamma = 1.0, 0.8
    nc, ne, _, _ = O.rank_update_f32(cores, diags, dC, dE, gamma, beta, lr)
    for a, c, g in zip(nc, cores, dC):
        np.testing.assert_allclose(a, c - lr * (g + 2 * beta * c), rtol=2e-6, atol=2e-6)
    pruned = 0
    for a, e, g in zip(ne, diags, dE):
        v = e - lr * g
        ref = O.soft_threshold(v, lr * gamma)
        far = np.abs(np.abs(v) - lr * gamma) > 1e-5
        np.testing.assert_allclose(a[far], ref[far], rtol=2e-6, atol=2e-6)
        assert np.all((a == 0)[far] == (np.abs(v) < lr * gamma)[far])
        pruned += int(np.sum(a == 0))
    assert pruned > 0  # the case exercises pruning


def test_rank_update_prunes_to_the_truncated_tt():
    """Entries the proximal step sets to zero drop their slices: the updated
    layer equals its rank-truncated TT."""
    rng = np.random.Generator(np.random.PCG64(13))
    shape = synth.LayerShape((2, 3), (3, 2), (1, 2, 3, 2, 1))
    cores, diags = _random_tt(rng, shape)
    dC = [np.zeros_like(c) for c in cores]
    dE = [np.zeros_like(e) for e in diags]
    # a threshold between the smallest and largest |D| entries
    allabs = np.sort(np.concatenate([np.abs(e) for e in diags]))
    lr, gamma = 1.0, float(allabs[len(allabs) // 2])
    nc, ne, _, _ = O.rank_update_f32(cores, diags, dC, dE, gamma, 0.0, lr)
    nc = [c.astype(np.float64) for c in nc]
    ne = [e.astype(np.float64) for e in ne]
    assert any(np.any(e == 0) for e in ne)
    tc, td, _ = O.truncate(nc, ne)
    x = rng.standard_normal((3, shape.N))
    d = len(shape.in_modes)
    np.testing.assert_allclose(O.dense_forward(nc, ne, d, x), O.dense_forward(tc, td, d, x),
                               rtol=1e-12, atol=1e-12)
