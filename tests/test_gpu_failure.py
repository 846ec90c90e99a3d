"""The device-side error path, exercised without a GPU fault.

Every wait in the kernels is bounded; when one runs out the kernel records
TT_ERR_TIMEOUT, stops its other warps, drains its own copies and MMAs, frees
its tensor memory and returns.  Here a test hook makes one arrival go missing
(the first CTA of one launch leaves a stage unloaded, or skips a grid-barrier
arrival) with the wait limit lowered to a few milliseconds, so the wait runs
out.  Each test checks that the call returns, that the status word reads
TT_ERR_TIMEOUT, and that the next ordinary call on the same device is correct.
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


@pytest.fixture
def short_limit():
    from tensor_train_compressed_tt_gb300 import ttc
    torch.cuda.synchronize()
    ttc.check(ttc.tt_set_wait_limit_ns(5_000_000), "tt_set_wait_limit_ns")   # 5 ms
    yield ttc
    torch.cuda.synchronize()
    ttc.check(ttc.tt_debug_skip_arrival(ttc.TT_DEBUG_NONE), "hook off")
    ttc.check(ttc.tt_set_wait_limit_ns(2_000_000_000), "tt_set_wait_limit_ns")


from parity_util import TOL, compare, gpu_layer, oracle_layer  # noqa: E402


def _layer_inputs(name, T, seed, **flags):
    from tensor_train_compressed_tt_gb300.layer import TTLinear
    w = synth.WORKLOADS[name]
    inp = synth.draw(w, seed=seed, tokens=T)
    s = w.layers[0]
    lay = TTLinear(s.in_modes, s.out_modes, s.ranks, torch.bfloat16, **flags)
    params = torch.from_numpy(synth.pack(inp.layers[0].cores, inp.layers[0].diags)).cuda()
    x = torch.from_numpy(inp.x).cuda().bfloat16()
    dy = torch.from_numpy(inp.dy).cuda().bfloat16()
    return w, inp, lay, params, x, dy


def _then_ordinary_call_is_correct(ttc):
    st = torch.cuda.current_stream().cuda_stream
    w = synth.WORKLOADS["tt768_bf16"]
    inp = synth.draw(w, seed=21, tokens=700)
    out = gpu_layer(w.layers[0], w.act, inp.layers[0], inp.x, inp.dy)
    compare(out, oracle_layer(w.layers[0], inp.layers[0], inp.x, inp.dy), TOL[w.act], "after")
    assert ttc.tt_get_device_status(st) == 0


@pytest.mark.parametrize("site,T", [("fwd", 128), ("fwd", 16384), ("bwd", 128), ("bwd", 16384)])
def test_token_kernel_wait_runs_out(short_limit, site, T):
    ttc = short_limit
    st = torch.cuda.current_stream().cuda_stream
    _, _, lay, params, x, dy = _layer_inputs("tt768_bf16", T, seed=20)
    ws = lay.workspace(T)
    if site == "bwd":
        lay.forward(x, params, ws=ws)
        torch.cuda.synchronize()
    ttc.check(ttc.tt_debug_skip_arrival(ttc.TT_DEBUG_FWD_TOKENS if site == "fwd"
                                        else ttc.TT_DEBUG_BWD_TOKENS), "hook")
    if site == "fwd":
        lay.forward(x, params, ws=ws)
    else:
        lay.backward(x, dy, params, ws=ws)
    assert ttc.tt_get_device_status(st) == 5   # TT_ERR_TIMEOUT, read and cleared
    assert ttc.tt_get_device_status(st) == 0
    _then_ordinary_call_is_correct(ttc)


@pytest.mark.parametrize("program", ["default", "deterministic", "rank_step"])
def test_merge_grid_barrier_wait_runs_out(short_limit, program):
    """Engine programs of more than one phase: the backward merge of an
    order-6 layer (two phases), its deterministic form (one phase a reverse
    step, then the first cores) and the backward merge with the rank-adaptive
    step (the step a phase of its own).  The first CTA skips a grid-barrier
    arrival and the others' waits run out."""
    ttc = short_limit
    st = torch.cuda.current_stream().cuda_stream
    det = program == "deterministic"
    _, _, lay, params, x, dy = _layer_inputs("tt768_bf16", 512, seed=22, deterministic=det)
    ws = lay.workspace(512)
    dx = torch.empty_like(x)
    dp = torch.empty_like(params)
    ttc.check(ttc.tt_debug_skip_arrival(ttc.TT_DEBUG_MERGE_BARRIER), "hook")
    if program != "rank_step":
        lay.backward(x, dy, params, dx=dx, dparams=dp, ws=ws)
    else:
        ttc.tt_backward_rank_update(lay.plan, 512, x.data_ptr(), dy.data_ptr(),
                                    params.data_ptr(), dx.data_ptr(), dp.data_ptr(), 0.01, 0.01,
                                    0.0, ws.data_ptr(), ws.numel(), st)
    assert ttc.tt_get_device_status(st) == 5
    _then_ordinary_call_is_correct(ttc)


def test_e4m3_forward_wait_runs_out(short_limit):
    """The E4M3 kernels' converter warps leave on the abort too."""
    from tensor_train_compressed_tt_gb300.layer import TTLinear
    ttc = short_limit
    st = torch.cuda.current_stream().cuda_stream
    w = synth.WORKLOADS["tt768_e4m3"]
    inp = synth.draw(w, seed=23, tokens=1000)
    s = w.layers[0]
    lay = TTLinear(s.in_modes, s.out_modes, s.ranks, torch.uint8)
    params = torch.from_numpy(synth.pack(inp.layers[0].cores, inp.layers[0].diags)).cuda()
    x = torch.from_numpy(synth.e4m3_bytes(inp.x)).cuda()
    dy = torch.from_numpy(synth.e4m3_bytes(inp.dy)).cuda()
    ws = lay.workspace(1000)
    ttc.check(ttc.tt_debug_skip_arrival(ttc.TT_DEBUG_BWD_TOKENS), "hook")
    lay.forward(x, params, ws=ws)
    lay.backward(x, dy, params, ws=ws)
    assert ttc.tt_get_device_status(st) == 5
    _then_ordinary_call_is_correct(ttc)


def test_wait_limit_arguments():
    from tensor_train_compressed_tt_gb300 import ttc
    assert ttc.tt_set_wait_limit_ns(10) == 1
    assert ttc.tt_debug_skip_arrival(-1) == 1
    assert ttc.tt_debug_skip_arrival(99) == 1
