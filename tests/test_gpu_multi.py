"""Several TT layers on one input (the Q, K and V projections of an encoder
block) through one multi-layer plan: every layer's y, dG_k and dD_k, and the
summed dx = sum_g dy_g W_g, against the oracle run layer by layer."""

import numpy as np
import pytest

from tensor_train_compressed_tt_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from tensor_train_compressed_tt_gb300 import _build
    _build.build()


from parity_util import TOL, TORCH_DT, compare, oracle_layer, to_dev  # noqa: E402


def _draw(shapes, T, seed, act):
    rng = np.random.Generator(np.random.PCG64(seed))
    lis = [synth.draw_layer(rng, sh, 0.05, "uniform") for sh in shapes]
    N = shapes[0].N
    x = rng.standard_normal((T, N)).astype(np.float32)
    dys = [rng.standard_normal((T, sh.M)).astype(np.float32) for sh in shapes]
    rnd = synth.round_e4m3 if act == "e4m3" else synth.round_bf16 if act == "bf16" else None
    if rnd is not None:
        x = rnd(x)
        dys = [rnd(d) for d in dys]
    return lis, x, dys


def _run(shapes, T, seed, act="bf16", **flags):
    from tensor_train_compressed_tt_gb300.layer import TTMulti
    lis, x, dys = _draw(shapes, T, seed, act)
    m = TTMulti([(s.in_modes, s.out_modes, s.ranks) for s in shapes], TORCH_DT[act], **flags)
    params = [torch.from_numpy(synth.pack(li.cores, li.diags)).cuda() for li in lis]
    xd = to_dev(x, act)
    dyd = [to_dev(d, act) for d in dys]
    ws = m.workspace(T)
    ys = m.forward(xd, params, ws=ws)
    dx, dps = m.backward(xd, dyd, params, ws=ws)
    torch.cuda.synchronize()
    return m, lis, x, dys, (xd, dyd, params, ws), ys, dx, dps


def _check(shapes, lis, x, dys, ys, dx, dps, tol):
    dx_ref = 0.0
    for g, sh in enumerate(shapes):
        ref = oracle_layer(sh, lis[g], x, dys[g])
        dx_ref = dx_ref + ref["dx"]
        gc, gd = synth.unpack(sh, dps[g].cpu().numpy())
        out = {"y": ys[g].float().cpu().numpy(), "dx": ref["dx"], "dcores": gc, "ddiags": gd}
        compare(out, ref, tol, f"layer {g}")
    from oracle import tt_oracle as O
    e = O.rel_err(dx.float().cpu().numpy(), dx_ref)
    assert e <= tol, f"summed dx: rel err {e:.3e}"


QKV = [synth.ENCODER_LAYERS[k] for k in ("q", "k", "v")]


@pytest.mark.parametrize("T,reuse_z", [(1000, False), (1000, True), (16384, False),
                                       (16384, True), (129, True), (1, False)])
def test_qkv_fused_against_oracle(T, reuse_z):
    _, lis, x, dys, _, ys, dx, dps = _run(QKV, T, seed=50 + T, reuse_z=reuse_z)
    _check(QKV, lis, x, dys, ys, dx, dps, TOL["bf16"])


def test_layers_of_different_widths():
    """Two layers with 768 and 3072 outputs on one x (different chunk counts
    per layer in the same kernel)."""
    shapes = [synth.ENCODER_LAYERS["q"], synth.ENCODER_LAYERS["up"]]
    _, lis, x, dys, _, ys, dx, dps = _run(shapes, 300, seed=61, reuse_z=True)
    _check(shapes, lis, x, dys, ys, dx, dps, TOL["bf16"])


def test_one_layer_multi_plan():
    shapes = [synth.ENCODER_LAYERS["o"]]
    _, lis, x, dys, _, ys, dx, dps = _run(shapes, 777, seed=62)
    _check(shapes, lis, x, dys, ys, dx, dps, TOL["bf16"])


def test_fused_forward_equals_single_layer_kernel():
    """Each y_g of the fused forward is bit for bit the single-layer
    forward's: the same tiles and the same MMA order per layer."""
    from tensor_train_compressed_tt_gb300.layer import TTLinear
    T = 5000
    m, lis, x, dys, (xd, dyd, params, ws), ys, dx, dps = _run(QKV, T, seed=63)
    for g, sh in enumerate(QKV):
        lay = TTLinear(sh.in_modes, sh.out_modes, sh.ranks, torch.bfloat16)
        y1 = lay.forward(xd, params[g])
        torch.cuda.synchronize()
        assert torch.equal(y1, ys[g]), g


def test_layer_by_layer_path():
    """f32 activations run the layers one after another and sum dx in layer
    order."""
    tiny = synth.WORKLOADS["tiny64_f32"].layers[0]
    shapes = [tiny] * 3
    _, lis, x, dys, _, ys, dx, dps = _run(shapes, 16, seed=64, act="f32")
    _check(shapes, lis, x, dys, ys, dx, dps, TOL["f32"])


@pytest.mark.parametrize("T", [1000, 20000])
def test_deterministic_fused(T):
    """TT_DETERMINISTIC on the fused Q/K/V kernels: per-CTA token-sum slots
    summed in CTA order, bit-reproducible, and the oracle's gradients.  20000
    tokens are more 128-token tiles than SMs (a second tile on some CTAs)."""
    m, lis, x, dys, (xd, dyd, params, ws), ys, dx, dps = _run(QKV, T, seed=65,
                                                              deterministic=True)
    _check(QKV, lis, x, dys, ys, dx, dps, TOL["bf16"])
    dx2, dps2 = m.backward(xd, dyd, params, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(dx, dx2)
    for a, b in zip(dps, dps2):
        assert torch.equal(a, b)


def test_e4m3_layers():
    shapes = [synth.ENCODER_LAYERS["q"], synth.ENCODER_LAYERS["k"]]
    _, lis, x, dys, _, ys, dx, dps = _run(shapes, 300, seed=66, act="e4m3")
    _check(shapes, lis, x, dys, ys, dx, dps, TOL["e4m3"])


def test_no_tokens_gives_zero_gradients():
    from tensor_train_compressed_tt_gb300.layer import TTMulti
    m = TTMulti([(s.in_modes, s.out_modes, s.ranks) for s in QKV], torch.bfloat16)
    lis, _, _ = _draw(QKV, 1, 67, "bf16")
    params = [torch.from_numpy(synth.pack(li.cores, li.diags)).cuda() for li in lis]
    x = torch.empty((0, 768), dtype=torch.bfloat16, device="cuda")
    dy = [torch.empty((0, 768), dtype=torch.bfloat16, device="cuda") for _ in QKV]
    dps = [torch.full((lay[2],), 7.0, device="cuda") for lay in m.layout]
    m.backward(x, dy, params, dparams=dps, ws=m.workspace(0))
    torch.cuda.synchronize()
    for t in dps:
        assert torch.count_nonzero(t).item() == 0
