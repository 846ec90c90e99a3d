"""GPU parity: libttc (through the C ABI) against the fp64 oracle.

Tolerances (norm-wise relative error per output tensor): 1e-4 for f32
activations, 2e-2 for bf16 or E4M3 activations with f32 accumulation; tensors whose
reference is exactly zero (pruned slices, removed layers) must be exactly 0.
"""

import dataclasses

import numpy as np
import pytest

from oracle import tt_oracle as O
from tensor_train_compressed_tt_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from tensor_train_compressed_tt_gb300 import _build
    _build.build()


from parity_util import (TOL, TORCH_DT, compare, gpu_ffn, gpu_layer, oracle_ffn,  # noqa: E402
                          oracle_layer, to_dev)


def _run(name, tokens=None, seed=0, reuse_z=False):
    w = synth.WORKLOADS[name]
    inp = synth.draw(w, seed=seed, tokens=tokens)
    shape = w.layers[0]
    out = gpu_layer(shape, w.act, inp.layers[0], inp.x, inp.dy, reuse_z=reuse_z)
    ref = oracle_layer(shape, inp.layers[0], inp.x, inp.dy)
    return compare(out, ref, TOL[w.act], f"{name} T={inp.x.shape[0]}")


def test_tiny64_f32():
    _run("tiny64_f32")


# Token counts cover the tile heights the host picks for one wave (16 .. 128
# tokens a tile) on 152 SMs: 16 (T <= 2432), 48 (6000), 80 (10000), 96
# (14000), and full 128-token tiles from three quarters of the SMs up (16384:
# 128 tiles, 18000: 141), each with a ragged last tile; two waves (112) run
# in the 1024 -> 4096 test at 32768 tokens.
@pytest.mark.parametrize("T", [1, 7, 128, 300, 6000, 10000, 14000, 16384, 18000])
def test_tt768_bf16(T):
    _run("tt768_bf16", tokens=T)


@pytest.mark.parametrize("name", ["pruned768_3072_bf16", "pruned768_768_bf16"])
def test_pruned_equals_truncated(name):
    _run(name)
    # and the truncated TT (slices removed) gives the same forward
    w = synth.WORKLOADS[name]
    inp = synth.draw(w, seed=0, tokens=257)
    shape = w.layers[0]
    tc, td, _ = O.truncate(inp.layers[0].cores, inp.layers[0].diags)
    tshape = synth.LayerShape(shape.in_modes, shape.out_modes,
                              tuple([1] + [len(e) for e in td] + [1]))
    # the truncated layer really is smaller: every link keeps nnz(D_k) ranks
    assert all(len(e) == np.count_nonzero(f) < f.size
               for e, f in zip(td, inp.layers[0].diags) if f.size > 1)
    out_t = gpu_layer(tshape, w.act, synth.LayerInputs(tc, td), inp.x, inp.dy)
    out_z = gpu_layer(shape, w.act, inp.layers[0], inp.x, inp.dy)
    assert O.rel_err(out_z["y"], out_t["y"]) <= TOL[w.act]
    assert O.rel_err(out_z["dx"], out_t["dx"]) <= TOL[w.act]


@pytest.mark.parametrize("T,reuse_z", [(4096, False), (16384, False), (32768, True)])
def test_tt1024_4096(T, reuse_z):
    """The 1024 -> 4096 rank-64 layer at each token count of its sweep, every
    output tensor (y, dx, each dG_k and dD_k) element by element against the
    oracle; 32768 tokens in the benchmark's launch configuration (kept z')."""
    _run("tt1024_4096_bf16", tokens=T, reuse_z=reuse_z)


@pytest.mark.parametrize("reuse_z,T", [(False, 1000), (True, 1000), (True, 16384)])
def test_ffn_pair(reuse_z, T):
    """The FFN pair against the oracle: y, dx and every dG_k, dD_k of both
    layers; 16384 tokens is the configured size, in the benchmark's launch
    configuration (the backward reusing the forward's work)."""
    w = synth.WORKLOADS["ffn768_3072_bf16"]
    inp = synth.draw(w, seed=0, tokens=T)
    out, gu, gd = gpu_ffn(w, inp, reuse_z=reuse_z)
    ref, ru, rd = oracle_ffn(w, inp)
    tol = TOL[w.act]
    assert O.rel_err(out["y"], ref["y"]) <= tol
    assert O.rel_err(out["dx"], ref["dx"]) <= tol
    for (a, b) in list(zip(gu[0], ru[0])) + list(zip(gd[0], rd[0])):
        assert O.rel_err(a, b) <= tol
    for (a, b) in list(zip(gu[1], ru[1])) + list(zip(gd[1], rd[1])):
        assert O.rel_err(a, b) <= tol


@pytest.mark.parametrize("d", [1, 2, 3, 4])
@pytest.mark.parametrize("act", ["f32", "bf16"])
def test_random_small_shapes(d, act):
    rng = np.random.Generator(np.random.PCG64(100 + d))
    for trial in range(4):
        shape = synth.random_shape(rng, d, max_mode=5, max_rank=6)
        li = synth.draw_layer(rng, shape, 0.5, "uniform" if trial % 2 else "pruned_half")
        T = int(rng.integers(1, 200))
        x = rng.standard_normal((T, shape.N)).astype(np.float32)
        dy = rng.standard_normal((T, shape.M)).astype(np.float32)
        if act == "bf16":
            x, dy = synth.round_bf16(x), synth.round_bf16(dy)
        out = gpu_layer(shape, act, li, x, dy)
        ref = oracle_layer(shape, li, x, dy)
        compare(out, ref, TOL[act], f"d={d} {shape} T={T}")


@pytest.mark.parametrize("reuse_z", [False, True])
def test_zero_tokens_backward_gives_zero_gradients(reuse_z):
    """T = 0: zero gradients, also with the reuse flags (a forward of no
    tokens leaves nothing to reuse)."""
    w = synth.WORKLOADS["tt768_bf16"]
    inp = synth.draw(w, seed=0, tokens=1)
    out = gpu_layer(w.layers[0], w.act, inp.layers[0], inp.x[:0], inp.dy[:0], reuse_z=reuse_z)
    assert out["y"].shape == (0, w.layers[0].M)
    assert all(np.all(g == 0) for g in out["dcores"])
    assert all(np.all(g == 0) for g in out["ddiags"])


def test_accumulate_flag_adds_into_dparams():
    import torch as th
    from tensor_train_compressed_tt_gb300.layer import TTLinear
    w = synth.WORKLOADS["tt768_bf16"]
    inp = synth.draw(w, seed=1, tokens=333)
    s = w.layers[0]
    params = th.from_numpy(synth.pack(inp.layers[0].cores, inp.layers[0].diags)).cuda()
    x = th.from_numpy(inp.x).cuda().bfloat16()
    dy = th.from_numpy(inp.dy).cuda().bfloat16()
    plain = TTLinear(s.in_modes, s.out_modes, s.ranks, th.bfloat16)
    _, g1 = plain.backward(x, dy, params)
    acc = TTLinear(s.in_modes, s.out_modes, s.ranks, th.bfloat16, accumulate=True)
    base = th.full_like(g1, 0.25)
    g2 = base.clone()
    acc.backward(x, dy, params, dparams=g2)
    th.cuda.synchronize()
    # the token sums are reduced with atomics, so the two runs may add in a
    # different order: compare norm-wise
    assert O.rel_err((g2 - base).cpu().numpy(), g1.cpu().numpy()) <= 1e-5


def test_all_zero_middle_link_removes_layer():
    w = synth.WORKLOADS["tt768_bf16"]
    inp = synth.draw(w, seed=2, tokens=200)
    li = inp.layers[0]
    li.diags[w.layers[0].d - 1][:] = 0.0
    out = gpu_layer(w.layers[0], w.act, li, inp.x, inp.dy)
    assert np.all(out["y"] == 0) and np.all(out["dx"] == 0)
    assert all(np.all(g == 0) for g in out["dcores"])
    assert all(np.all(g == 0) for g in out["ddiags"])


def test_full_size_identities_tt1024_4096():
    """At 32768 tokens: <x,dx> = <G_k,dG_k> = <D_k,dD_k> = <dy,y> for every k."""
    w = synth.WORKLOADS["tt1024_4096_bf16"]
    inp = synth.draw(w, seed=0)
    shape = w.layers[0]
    out = gpu_layer(shape, w.act, inp.layers[0], inp.x, inp.dy)
    ref = float(np.sum(out["y"].astype(np.float64) * inp.dy))
    scale = float(np.linalg.norm(out["y"])) * float(np.linalg.norm(inp.dy))
    # bf16 rounding of y and dx bounds how well the products can agree
    assert abs(float(np.sum(inp.x.astype(np.float64) * out["dx"])) - ref) <= 2e-2 * scale
    for c, g in zip(inp.layers[0].cores, out["dcores"]):
        assert abs(float(np.sum(c.astype(np.float64) * g)) - ref) <= 2e-2 * scale
    for e, g in zip(inp.layers[0].diags, out["ddiags"]):
        assert abs(float(np.sum(e.astype(np.float64) * g)) - ref) <= 2e-2 * scale
    # sampled rows of y and dx against the oracle, one token at a time
    rows = np.random.default_rng(0).choice(inp.x.shape[0], 64, replace=False)
    sub = oracle_layer(shape, inp.layers[0], inp.x[rows], inp.dy[rows])
    assert O.rel_err(out["y"][rows], sub["y"]) <= TOL[w.act]
    assert O.rel_err(out["dx"][rows], sub["dx"]) <= TOL[w.act]


@pytest.mark.parametrize("name", ["tt768_bf16", "pruned768_3072_bf16", "tiny64_f32",
                                  "tt768_e4m3"])
def test_reuse_merge_matches_default(name):
    """TT_REUSE_MERGE: backward after forward on the same workspace, twice."""
    import torch as th
    from tensor_train_compressed_tt_gb300.layer import TTLinear
    w = synth.WORKLOADS[name]
    inp = synth.draw(w, seed=3, tokens=min(w.tokens, 700))
    s = w.layers[0]
    dt = TORCH_DT[w.act]
    params = th.from_numpy(synth.pack(inp.layers[0].cores, inp.layers[0].diags)).cuda()
    x = to_dev(inp.x, w.act)
    dy = to_dev(inp.dy, w.act)
    ref = TTLinear(s.in_modes, s.out_modes, s.ranks, dt)
    y0 = ref.forward(x, params)
    dx0, g0 = ref.backward(x, dy, params)
    reu = TTLinear(s.in_modes, s.out_modes, s.ranks, dt, reuse_merge=True)
    ws = reu.workspace(x.shape[0])
    for _ in range(2):
        y1 = reu.forward(x, params, ws=ws)
        dx1, g1 = reu.backward(x, dy, params, ws=ws)
        dx2, g2 = reu.backward(x, dy, params, ws=ws)   # a second backward reuses again
        th.cuda.synchronize()
        assert th.equal(y0, y1)
        assert th.equal(dx0, dx1) and th.equal(dx0, dx2)
        # atomically reduced token sums: equal up to summation order
        assert O.rel_err(g1.cpu().numpy(), g0.cpu().numpy()) <= 1e-5
        assert O.rel_err(g2.cpu().numpy(), g0.cpu().numpy()) <= 1e-5


def test_internal_rank_above_64_uses_generic_merge():
    """A link rank above 64 takes the generic (GEMM-phase) merge program."""
    rng = np.random.Generator(np.random.PCG64(77))
    for shape, act in [(synth.LayerShape((4, 3, 2), (2, 3, 4), (1, 4, 70, 6, 66, 4, 1)), "f32"),
                       (synth.LayerShape((16, 8), (8, 16), (1, 16, 40, 72, 1)), "bf16")]:
        li = synth.draw_layer(rng, shape, 0.3, "uniform")
        T = 77
        x = rng.standard_normal((T, shape.N)).astype(np.float32)
        dy = rng.standard_normal((T, shape.M)).astype(np.float32)
        if act == "bf16":
            x, dy = synth.round_bf16(x), synth.round_bf16(dy)
        compare(gpu_layer(shape, act, li, x, dy), oracle_layer(shape, li, x, dy), TOL[act],
                f"{shape}")


# ---- E4M3 activations ------------------------------------------------------

@pytest.mark.parametrize("T", [1, 7, 300, 10000, 16384])
def test_tt768_e4m3(T):
    _run("tt768_e4m3", tokens=T)


def test_tt1024_4096_e4m3():
    _run("tt1024_4096_e4m3", tokens=4096)


@pytest.mark.parametrize("name,T", [("tt768_e4m3", 1000), ("tt1024_4096_e4m3", 777)])
def test_e4m3_equals_bf16_kernels_on_the_same_values(name, T):
    """E4M3 values are exact in bf16, so the E4M3 kernels, which widen the tile
    in shared memory, must give the bf16 kernels' y and dx bit for bit on the
    same values (dparams: equal up to the order of the atomic token sums)."""
    import torch as th
    from tensor_train_compressed_tt_gb300.layer import TTLinear
    w = synth.WORKLOADS[name]
    inp = synth.draw(w, seed=5, tokens=T)
    s = w.layers[0]
    params = th.from_numpy(synth.pack(inp.layers[0].cores, inp.layers[0].diags)).cuda()
    outs = []
    for act in ("e4m3", "bf16"):
        lay = TTLinear(s.in_modes, s.out_modes, s.ranks, TORCH_DT[act])
        x, dy = to_dev(inp.x, act), to_dev(inp.dy, act)
        y = lay.forward(x, params)
        dx, g = lay.backward(x, dy, params)
        th.cuda.synchronize()
        outs.append((y, dx, g))
    (y8, dx8, g8), (yb, dxb, gb) = outs
    assert y8.dtype == th.bfloat16 and dx8.dtype == th.bfloat16
    assert th.equal(y8, yb)
    assert th.equal(dx8, dxb)
    assert O.rel_err(g8.cpu().numpy(), gb.cpu().numpy()) <= 1e-5


def test_full_size_e4m3_tt1024_4096():
    """The benchmarked E4M3 configuration at its full 32768 tokens: the
    <x,dx> = <G_k,dG_k> = <D_k,dD_k> = <dy,y> identities, and sampled rows of
    y and dx against the oracle one token at a time."""
    w = synth.WORKLOADS["tt1024_4096_e4m3"]
    inp = synth.draw(w, seed=0)
    shape = w.layers[0]
    out = gpu_layer(shape, w.act, inp.layers[0], inp.x, inp.dy)
    ref = float(np.sum(out["y"].astype(np.float64) * inp.dy))
    scale = float(np.linalg.norm(out["y"])) * float(np.linalg.norm(inp.dy))
    assert abs(float(np.sum(inp.x.astype(np.float64) * out["dx"])) - ref) <= 2e-2 * scale
    for c, g in zip(inp.layers[0].cores, out["dcores"]):
        assert abs(float(np.sum(c.astype(np.float64) * g)) - ref) <= 2e-2 * scale
    for e, g in zip(inp.layers[0].diags, out["ddiags"]):
        assert abs(float(np.sum(e.astype(np.float64) * g)) - ref) <= 2e-2 * scale
    rows = np.random.default_rng(1).choice(inp.x.shape[0], 64, replace=False)
    sub = oracle_layer(shape, inp.layers[0], inp.x[rows], inp.dy[rows])
    assert O.rel_err(out["y"][rows], sub["y"]) <= TOL[w.act]
    assert O.rel_err(out["dx"][rows], sub["dx"]) <= TOL[w.act]


def test_tt768_e4m3_pruned():
    """E4M3 inputs with half of every D_k exactly zero (compacted middle rank)."""
    w = synth.WORKLOADS["tt768_e4m3"]
    import dataclasses
    wp = dataclasses.replace(w, diag="pruned_half")
    inp = synth.draw(wp, seed=2, tokens=2000)
    shape = wp.layers[0]
    out = gpu_layer(shape, wp.act, inp.layers[0], inp.x, inp.dy)
    ref = oracle_layer(shape, inp.layers[0], inp.x, inp.dy)
    compare(out, ref, TOL["e4m3"], "tt768 e4m3 pruned")


# ---- TT_REUSE_Z: the backward reads the forward's z' -----------------------

@pytest.mark.parametrize("name,T", [("tt768_bf16", 16384), ("tt768_e4m3", 16384),
                                    ("tt768_bf16", 300), ("pruned768_3072_bf16", 1000),
                                    ("tt1024_4096_bf16", 4096), ("tt1024_4096_e4m3", 777)])
def test_reuse_z_against_oracle(name, T):
    """Every output against the oracle, element by element, at the benchmark's
    launch configuration (kept z') and full token count where listed."""
    _run(name, tokens=T, reuse_z=True)


@pytest.mark.parametrize("name", ["tt768_bf16", "tt768_e4m3", "pruned768_768_bf16"])
def test_reuse_z_matches_recompute(name):
    """y and dx are the recomputing path's bit for bit (the same z' tile feeds
    the same MMAs); dparams agree to rounding: dD_d is summed from the bf16 z'
    divided by D_d instead of the f32 z.  Two backward calls after one forward
    read the same kept z'."""
    import torch as th
    from tensor_train_compressed_tt_gb300.layer import TTLinear
    w = synth.WORKLOADS[name]
    inp = synth.draw(w, seed=4, tokens=1000)
    s = w.layers[0]
    params = th.from_numpy(synth.pack(inp.layers[0].cores, inp.layers[0].diags)).cuda()
    x, dy = to_dev(inp.x, w.act), to_dev(inp.dy, w.act)
    ref = TTLinear(s.in_modes, s.out_modes, s.ranks, TORCH_DT[w.act])
    y0 = ref.forward(x, params)
    dx0, g0 = ref.backward(x, dy, params)
    kz = TTLinear(s.in_modes, s.out_modes, s.ranks, TORCH_DT[w.act], reuse_z=True)
    assert kz.workspace_bytes(1000) >= ref.workspace_bytes(1000) + 1000 * 128
    ws = kz.workspace(1000)
    y1 = kz.forward(x, params, ws=ws)
    dx1, g1 = kz.backward(x, dy, params, ws=ws)
    dx2, g2 = kz.backward(x, dy, params, ws=ws)
    th.cuda.synchronize()
    assert th.equal(y0, y1)
    assert th.equal(dx0, dx1) and th.equal(dx0, dx2)
    a0 = g0.cpu().numpy()
    assert O.rel_err(g1.cpu().numpy(), a0) <= 1e-3
    assert O.rel_err(g2.cpu().numpy(), g1.cpu().numpy()) <= 1e-5


def test_ffn_reuse_matches_recompute():
    """FFN with the forward's merges, z', h and GELU(h) kept: y and dx are the
    recomputing path's bit for bit; dparams agree to rounding; a second
    backward after one forward gives the same."""
    import torch as th
    from tensor_train_compressed_tt_gb300.layer import TTFFN
    w = synth.WORKLOADS["ffn768_3072_bf16"]
    inp = synth.draw(w, seed=6, tokens=700)
    up, dn = w.layers
    pu = th.from_numpy(synth.pack(inp.layers[0].cores, inp.layers[0].diags)).cuda()
    pd = th.from_numpy(synth.pack(inp.layers[1].cores, inp.layers[1].diags)).cuda()
    x, dy = to_dev(inp.x, w.act), to_dev(inp.dy, w.act)
    outs = []
    for keep in (False, True):
        f = TTFFN((up.in_modes, up.out_modes, up.ranks), (dn.in_modes, dn.out_modes, dn.ranks),
                  TORCH_DT[w.act], reuse_z=keep)
        ws = f.workspace(700)
        y = f.forward(x, pu, pd, ws=ws)
        dx, gu, gd = f.backward(x, dy, pu, pd, ws=ws)
        dx2, gu2, gd2 = f.backward(x, dy, pu, pd, ws=ws)
        th.cuda.synchronize()
        assert th.equal(dx, dx2)
        assert O.rel_err(gu2.cpu().numpy(), gu.cpu().numpy()) <= 1e-5
        outs.append((y, dx, gu, gd))
    (y0, dx0, gu0, gd0), (y1, dx1, gu1, gd1) = outs
    assert th.equal(y0, y1) and th.equal(dx0, dx1)
    assert O.rel_err(gu1.cpu().numpy(), gu0.cpu().numpy()) <= 1e-3
    assert O.rel_err(gd1.cpu().numpy(), gd0.cpu().numpy()) <= 1e-3


@pytest.mark.parametrize("T,reuse_z", [(1, True), (127, False), (129, True)])
def test_ffn_pair_edge_token_counts(T, reuse_z):
    """The fused FFN kernels on one token, on one token short of a 128-token
    tile and one past it: y, dx and every gradient of both layers."""
    w = synth.WORKLOADS["ffn768_3072_bf16"]
    inp = synth.draw(w, seed=21 + T, tokens=T)
    out, gu, gd = gpu_ffn(w, inp, reuse_z=reuse_z)
    ref, ru, rd = oracle_ffn(w, inp)
    tol = TOL[w.act]
    assert O.rel_err(out["y"], ref["y"]) <= tol
    assert O.rel_err(out["dx"], ref["dx"]) <= tol
    for (a, b) in (list(zip(gu[0], ru[0])) + list(zip(gd[0], rd[0])) + list(zip(gu[1], ru[1])) +
                   list(zip(gd[1], rd[1]))):
        assert O.rel_err(a, b) <= tol


@pytest.mark.parametrize("reuse_z", [False, True])
def test_ffn_pair_zero_tokens(reuse_z):
    """T = 0 through the FFN plan: y is empty and every gradient exactly 0."""
    w = synth.WORKLOADS["ffn768_3072_bf16"]
    inp = synth.draw(w, seed=0, tokens=1)
    inp0 = dataclasses.replace(inp, x=inp.x[:0], dy=inp.dy[:0])
    out, gu, gd = gpu_ffn(w, inp0, reuse_z=reuse_z)
    assert out["y"].shape == (0, w.layers[1].M)
    for g in list(gu[0]) + list(gu[1]) + list(gd[0]) + list(gd[1]):
        assert np.all(g == 0)


@pytest.mark.parametrize("act,rmid", [("f32", 12), ("bf16", 12), ("bf16", 40)])
def test_ffn_pair_small(act, rmid):
    """A small FFN pair on both token paths (f32: SIMT GEMMs and the f32 GELU
    kernels; bf16: tensor-core kernels), 300 tokens, against the oracle.  A
    middle rank of 12 takes the fused kernels' 32-wide rank products, 40 the
    64-wide ones."""
    import dataclasses
    up = synth.LayerShape((8, 16), (16, 16), (1, 8, rmid, 16, 1))
    dn = synth.LayerShape((16, 16), (8, 16), (1, 16, rmid, 8, 1))
    w = dataclasses.replace(synth.WORKLOADS["ffn768_3072_bf16"], name=f"ffn_small_{act}_{rmid}",
                            layers=(up, dn), tokens=300, act=act, core_std=0.2)
    inp = synth.draw(w, seed=8)
    out, gu, gd = gpu_ffn(w, inp)
    ref, ru, rd = oracle_ffn(w, inp)
    tol = TOL[act]
    assert O.rel_err(out["y"], ref["y"]) <= tol
    assert O.rel_err(out["dx"], ref["dx"]) <= tol
    for (a, b) in list(zip(gu[0], ru[0])) + list(zip(gd[0], rd[0])):
        assert O.rel_err(a, b) <= tol
    for (a, b) in list(zip(gu[1], ru[1])) + list(zip(gd[1], rd[1])):
        assert O.rel_err(a, b) <= tol
