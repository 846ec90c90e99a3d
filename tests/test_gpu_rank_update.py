"""GPU parity of the rank-adaptive step (tt_rank_update) against the oracle.

The step is elementwise float32 arithmetic in a fixed order without fused
multiply-adds, and the oracle applies the same operations in numpy float32,
so the comparison is bit for bit (including which diagonal entries become
exactly zero).
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


from parity_util import TOL, compare, gpu_layer, oracle_layer  # noqa: E402


def _bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def _case(name, seed):
    from tensor_train_compressed_tt_gb300.layer import TTLinear
    w = synth.WORKLOADS[name]
    s = w.layers[0]
    rng = np.random.Generator(np.random.PCG64(seed))
    li = synth.draw(w, seed=seed, tokens=1).layers[0]
    dC = [rng.standard_normal(c.shape).astype(np.float32) for c in li.cores]
    dE = [np.where(e != 0, rng.standard_normal(e.shape), 0.0).astype(np.float32) for e in li.diags]
    layer = TTLinear(s.in_modes, s.out_modes, s.ranks, torch.float32)
    return w, s, li, dC, dE, layer


@pytest.mark.parametrize("name", ["tt768_bf16", "pruned768_3072_bf16", "tiny64_f32",
                                  "tt1024_4096_bf16"])
@pytest.mark.parametrize("gamma,beta,lr", [(0.05, 0.01, 0.0), (0.3, 0.02, 1.0), (0.0, 0.0, 0.25)])
def test_rank_update_bit_exact(name, gamma, beta, lr):
    w, s, li, dC, dE, layer = _case(name, 21)
    p = torch.from_numpy(synth.pack(li.cores, li.diags)).cuda()
    g = torch.from_numpy(synth.pack(dC, dE)).cuda()
    layer.rank_update(p, g, gamma, beta, lr)
    torch.cuda.synchronize()
    oc, od, odc, odd = O.rank_update_f32(li.cores, li.diags, dC, dE, gamma, beta, lr)
    ref_p = synth.pack(oc, od)
    ref_g = synth.pack(odc, odd)
    assert np.array_equal(_bits(p.cpu().numpy()), _bits(ref_p))
    assert np.array_equal(_bits(g.cpu().numpy()), _bits(ref_g))
    if lr > 0 and gamma * lr >= 0.3:
        assert sum(int(np.sum(e == 0)) for e in od) > 0  # the step pruned entries


def test_pruned_by_the_step_equals_truncated_tt():
    """A proximal step that zeroes diagonal entries; the next forward and
    backward equal the oracle and the rank-truncated layer."""
    w, s, li, dC, dE, _ = _case("tt768_bf16", 22)
    from tensor_train_compressed_tt_gb300.layer import TTLinear
    layer = TTLinear(s.in_modes, s.out_modes, s.ranks, torch.bfloat16)
    p = torch.from_numpy(synth.pack(li.cores, li.diags)).cuda()
    g = torch.from_numpy(synth.pack(dC, dE)).cuda()
    layer.rank_update(p, g, 0.6, 0.0, 1.0)   # threshold 0.6: prunes part of D ~ U(0.5, 1.5)
    torch.cuda.synchronize()
    cores, diags = synth.unpack(s, p.cpu().numpy())
    nz = [int(np.sum(e == 0)) for e in diags]
    assert sum(nz) > 0 and all(n < len(e) for n, e in zip(nz, diags))
    upd = synth.LayerInputs(cores, diags)
    inp = synth.draw(w, seed=5, tokens=300)
    out = gpu_layer(s, w.act, upd, inp.x, inp.dy)
    compare(out, oracle_layer(s, upd, inp.x, inp.dy), TOL[w.act], "after the rank step")
    tc, td, _ = O.truncate(cores, diags)
    ts = synth.LayerShape(s.in_modes, s.out_modes, tuple([1] + [len(e) for e in td] + [1]))
    out_t = gpu_layer(ts, w.act, synth.LayerInputs(tc, td), inp.x, inp.dy)
    assert O.rel_err(out["y"], out_t["y"]) <= TOL[w.act]
    assert O.rel_err(out["dx"], out_t["dx"]) <= TOL[w.act]


@pytest.mark.parametrize("name,T", [("tt768_bf16", 2000), ("pruned768_3072_bf16", 700),
                                    ("tiny64_f32", 16), ("tt1024_4096_bf16", 1000)])
@pytest.mark.parametrize("gamma,beta,lr", [(0.05, 0.01, 0.0), (0.6, 0.02, 1.0)])
def test_backward_with_fused_rank_step_equals_the_two_calls(name, T, gamma, beta, lr):
    """tt_backward_rank_update (the step as the last phase of the backward's
    merge program) gives the bits of tt_backward then tt_rank_update, and its
    step is the oracle's float32 step on the gradients it produced.  The
    plans are deterministic, so the two backward passes sum in one order."""
    from tensor_train_compressed_tt_gb300 import ttc
    from parity_util import TORCH_DT, to_dev
    w = synth.WORKLOADS[name]
    s = w.layers[0]
    inp = synth.draw(w, seed=31, tokens=T)
    act = {"bf16": ttc.TT_DT_BF16, "f32": ttc.TT_DT_F32}[w.act]
    plan = ttc.tt_plan(ttc.make_desc(s.in_modes, s.out_modes, s.ranks, act,
                                     ttc.TT_DETERMINISTIC))
    x, dy = to_dev(inp.x, w.act), to_dev(inp.dy, w.act)
    p0 = torch.from_numpy(synth.pack(inp.layers[0].cores, inp.layers[0].diags)).cuda()
    st = torch.cuda.current_stream().cuda_stream
    ws = torch.empty(ttc.tt_workspace_size(plan, T), dtype=torch.uint8, device="cuda")
    outs = []
    for fused in (False, True):
        p = p0.clone()
        g = torch.empty_like(p0)
        dx = torch.empty((T, s.N), dtype=TORCH_DT[w.act], device="cuda")
        if fused:
            ttc.check(ttc.tt_backward_rank_update(plan, T, x.data_ptr(), dy.data_ptr(),
                                                  p.data_ptr(), dx.data_ptr(), g.data_ptr(),
                                                  gamma, beta, lr, ws.data_ptr(), ws.numel(), st))
        else:
            ttc.check(ttc.tt_backward(plan, T, x.data_ptr(), dy.data_ptr(), p.data_ptr(),
                                      dx.data_ptr(), g.data_ptr(), ws.data_ptr(), ws.numel(), st))
            grad = g.clone()
            ttc.check(ttc.tt_rank_update(plan, p.data_ptr(), g.data_ptr(), gamma, beta, lr, st))
        torch.cuda.synchronize()
        outs.append((p, g, dx))
    (p1, g1, dx1), (p2, g2, dx2) = outs
    assert torch.equal(dx1, dx2)
    assert torch.equal(p1, p2) and torch.equal(g1, g2)
    # the step itself against the oracle, on the gradients the backward produced
    gc, gd = synth.unpack(s, grad.cpu().numpy())
    oc, od, odc, odd = O.rank_update_f32(inp.layers[0].cores, inp.layers[0].diags, gc, gd,
                                         gamma, beta, lr)
    assert np.array_equal(_bits(p2.cpu().numpy()), _bits(synth.pack(oc, od)))
    assert np.array_equal(_bits(g2.cpu().numpy()), _bits(synth.pack(odc, odd)))
    assert ttc.tt_get_device_status(st) == 0
