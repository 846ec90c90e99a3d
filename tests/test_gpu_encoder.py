"""The TT layers of one encoder block (Q, K, V, O and the GELU FFN pair) as
one step, eager and replayed from one CUDA graph: every layer's y, dx, dG_k
and dD_k against the oracle."""

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


from parity_util import TOL, compare, oracle_layer  # noqa: E402


def _f64(li):
    return ([c.astype(np.float64) for c in li.cores], [e.astype(np.float64) for e in li.diags])


def _block(T, seed, fuse_qkv=True):
    from tensor_train_compressed_tt_gb300.encoder import PROJ, TTEncoderBlock
    inp = synth.draw_encoder(T, seed)
    blk = TTEncoderBlock(fuse_qkv=fuse_qkv)
    dev = lambda a: torch.from_numpy(a).cuda().bfloat16()  # noqa: E731
    x, xo, xf = dev(inp.x), dev(inp.xo), dev(inp.xf)
    dy = {k: dev(v) for k, v in inp.dy.items()}
    params = {nm: torch.from_numpy(synth.pack(li.cores, li.diags)).cuda()
              for nm, li in inp.layers.items()}
    b = blk.buffers(T)
    return inp, blk, (x, xo, xf, dy, params), b, PROJ


def _check(inp, b, PROJ):
    """Every layer's y and gradients; dx per input (dx_qkv: the summed dx of
    Q, K and V, when they run fused)."""
    L = synth.ENCODER_LAYERS
    xin = {"q": inp.x, "k": inp.x, "v": inp.x, "o": inp.xo}
    dx_sum = 0.0
    for nm in PROJ:
        ref = oracle_layer(L[nm], inp.layers[nm], xin[nm], inp.dy[nm])
        if nm != "o":
            dx_sum = dx_sum + ref["dx"]
        gc, gd = synth.unpack(L[nm], b[f"dp_{nm}"].cpu().numpy())
        dx = b[f"dx_{nm}"].float().cpu().numpy() if f"dx_{nm}" in b else ref["dx"]
        out = {"y": b[f"y_{nm}"].float().cpu().numpy(), "dx": dx, "dcores": gc, "ddiags": gd}
        compare(out, ref, TOL["bf16"], f"layer {nm}")
    if "dx_qkv" in b:
        assert O.rel_err(b["dx_qkv"].float().cpu().numpy(), dx_sum) <= TOL["bf16"]
    up, dn = _f64(inp.layers["up"]), _f64(inp.layers["down"])
    y = O.ffn_forward(up, dn, 3, 3, inp.xf)
    dx, gu, gdn = O.ffn_backward(up, dn, 3, 3, inp.xf, inp.dy["ffn"])
    assert O.rel_err(b["y_ffn"].float().cpu().numpy(), y) <= TOL["bf16"]
    assert O.rel_err(b["dx_ffn"].float().cpu().numpy(), dx) <= TOL["bf16"]
    for key, shape, ref in (("dp_up", L["up"], gu), ("dp_down", L["down"], gdn)):
        gc, gd = synth.unpack(shape, b[key].cpu().numpy())
        for a, r in list(zip(gc, ref[0])) + list(zip(gd, ref[1])):
            assert O.rel_err(a, r) <= TOL["bf16"], key


@pytest.mark.parametrize("T,fuse_qkv", [(300, True), (4096, True), (1000, False)])
def test_encoder_block_step_against_oracle(T, fuse_qkv):
    inp, blk, args, b, PROJ = _block(T, seed=40, fuse_qkv=fuse_qkv)
    blk.step(*args, b)
    torch.cuda.synchronize()
    _check(inp, b, PROJ)


def test_encoder_block_graph_replay_matches_eager():
    """One CUDA graph holds the whole block; its replay gives the eager
    step's y and dx bit for bit and the oracle's gradients."""
    T = 1000
    inp, blk, args, b, PROJ = _block(T, seed=41)
    blk.step(*args, b)
    torch.cuda.synchronize()
    eager = {k: v.clone() for k, v in b.items() if k.startswith(("y_", "dx_"))}
    for k in b:
        if k.startswith(("y_", "dx_", "dp_")):
            b[k].zero_()
    g = blk.capture(T, *args, b)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for k, v in eager.items():
        assert torch.equal(b[k], v), k
    _check(inp, b, PROJ)
