"""TT_DETERMINISTIC: the same inputs give bit-identical dx and dparams.

Without the flag the token sums and the merge backward's K splits are added
with atomics in whatever order the CTAs reach them, so repeated backward
calls agree only to rounding.  With it every sum over tokens is taken in a
fixed order (per-CTA slots summed in CTA order, no atomic K splits), so two
runs must agree bit for bit, and the results must still match the oracle.
"""

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


from parity_util import TOL, TORCH_DT, oracle_layer, to_dev  # noqa: E402


def _runs(name, T, reuse_z, seed=11, runs=3):
    from tensor_train_compressed_tt_gb300.layer import TTLinear
    w = synth.WORKLOADS[name]
    inp = synth.draw(w, seed=seed, tokens=T)
    s = w.layers[0]
    params = torch.from_numpy(synth.pack(inp.layers[0].cores, inp.layers[0].diags)).cuda()
    x, dy = to_dev(inp.x, w.act), to_dev(inp.dy, w.act)
    lay = TTLinear(s.in_modes, s.out_modes, s.ranks, TORCH_DT[w.act], reuse_z=reuse_z,
                   deterministic=True)
    ws = lay.workspace(T)
    outs = []
    for _ in range(runs):
        y = lay.forward(x, params, ws=ws)
        dx, g = lay.backward(x, dy, params, ws=ws)
        torch.cuda.synchronize()
        outs.append((y.clone(), dx.clone(), g.clone()))
    return w, s, inp, outs


@pytest.mark.parametrize("name,T,reuse_z", [("tt768_bf16", 16384, True), ("tt768_bf16", 777, False),
                                            ("tt768_e4m3", 3000, True),
                                            ("tt1024_4096_bf16", 32768, True),
                                            ("pruned768_3072_bf16", 1000, False),
                                            ("tiny64_f32", 16, False)])
def test_bit_identical_runs_and_oracle_parity(name, T, reuse_z):
    w, s, inp, outs = _runs(name, T, reuse_z)
    y0, dx0, g0 = outs[0]
    for y, dx, g in outs[1:]:
        assert torch.equal(y, y0)
        assert torch.equal(dx, dx0)
        assert torch.equal(g, g0), "dparams differ between two deterministic runs"
    # and the result is the right one
    ref = oracle_layer(s, inp.layers[0], inp.x, inp.dy)
    gc, gd = synth.unpack(s, g0.cpu().numpy())
    tol = TOL[w.act]
    assert O.rel_err(dx0.float().cpu().numpy(), ref["dx"]) <= tol
    for a, b in zip(gc, ref["dcores"]):
        assert O.rel_err(a, b) <= tol
    for a, b in zip(gd, ref["ddiags"]):
        assert O.rel_err(a, b) <= tol
        assert np.all(a[np.asarray(b) == 0.0] == 0.0)


def test_f32_token_path_is_bit_identical():
    """An f32 layer too large for the single-CTA path (SIMT token kernels)."""
    from tensor_train_compressed_tt_gb300.layer import TTLinear
    rng = np.random.Generator(np.random.PCG64(5))
    shape = synth.LayerShape((8, 8, 8), (8, 8, 8), (1, 8, 16, 16, 16, 8, 1))
    li = synth.draw_layer(rng, shape, 0.3, "uniform")
    T = 6000
    x = rng.standard_normal((T, shape.N)).astype(np.float32)
    dy = rng.standard_normal((T, shape.M)).astype(np.float32)
    params = torch.from_numpy(synth.pack(li.cores, li.diags)).cuda()
    lay = TTLinear(shape.in_modes, shape.out_modes, shape.ranks, torch.float32,
                   deterministic=True)
    xd, dyd = torch.from_numpy(x).cuda(), torch.from_numpy(dy).cuda()
    res = [lay.backward(xd, dyd, params) for _ in range(3)]
    torch.cuda.synchronize()
    for dx, g in res[1:]:
        assert torch.equal(dx, res[0][0]) and torch.equal(g, res[0][1])
    ref = oracle_layer(shape, li, x, dy)
    gc, gd = synth.unpack(shape, res[0][1].cpu().numpy())
    for a, b in list(zip(gc, ref["dcores"])) + list(zip(gd, ref["ddiags"])):
        assert O.rel_err(a, b) <= 1e-4


@pytest.mark.parametrize("T", [2000, 20000])
def test_ffn_pair_is_bit_identical(T):
    """The fused FFN kernels with per-CTA slots: bit-identical runs, and the
    oracle's gradients.  20000 tokens are more 128-token tiles than SMs, so
    some CTAs add a second tile into their slots."""
    from tensor_train_compressed_tt_gb300.layer import TTFFN
    from parity_util import oracle_ffn
    w = synth.WORKLOADS["ffn768_3072_bf16"]
    inp = synth.draw(w, seed=3, tokens=T)
    up, dn = w.layers
    pu = torch.from_numpy(synth.pack(inp.layers[0].cores, inp.layers[0].diags)).cuda()
    pd = torch.from_numpy(synth.pack(inp.layers[1].cores, inp.layers[1].diags)).cuda()
    x, dy = to_dev(inp.x, w.act), to_dev(inp.dy, w.act)
    f = TTFFN((up.in_modes, up.out_modes, up.ranks), (dn.in_modes, dn.out_modes, dn.ranks),
              TORCH_DT[w.act], reuse_z=True, deterministic=True)
    ws = f.workspace(T)
    res = []
    for _ in range(3):
        y = f.forward(x, pu, pd, ws=ws).clone()
        res.append((y,) + tuple(t.clone() for t in f.backward(x, dy, pu, pd, ws=ws)))
    torch.cuda.synchronize()
    for r in res[1:]:
        assert all(torch.equal(a, b) for a, b in zip(r, res[0]))
    y, dx, gu, gd = res[0]
    ref, ru, rd = oracle_ffn(w, inp)
    tol = TOL[w.act]
    assert O.rel_err(y.float().cpu().numpy(), ref["y"]) <= tol
    assert O.rel_err(dx.float().cpu().numpy(), ref["dx"]) <= tol
    for sh, g, r in ((up, gu, ru), (dn, gd, rd)):
        gc, gdg = synth.unpack(sh, g.cpu().numpy())
        for a, b in list(zip(gc, r[0])) + list(zip(gdg, r[1])):
            assert O.rel_err(a, b) <= tol
