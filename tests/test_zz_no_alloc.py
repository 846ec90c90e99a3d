"""tt_forward_noalloc: the forward for callers that cannot allocate device memory.

Such callers (a plain-C host or plugin without a device allocator, or a
process that must not call cudaMalloc once running) get the scratch from a
fixed device array inside the library instead of a caller workspace.  The
no-alloc call runs the very same kernels on the same inputs as tt_forward,
so its output must equal tt_forward's bit for bit; a stale or partly
overwritten scratch would show up as a difference.  This file is collected
last on purpose, so that a failure here cannot hide the result of any other
test; it must also pass when run on its own.
"""

import numpy as np
import pytest

from tensor_train_compressed_tt_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.mark.parametrize("name,T,keep_z", [("tt768_bf16", 300, False), ("tiny64_f32", 16, False),
                                            ("tt1024_4096_bf16", 257, False),
                                            ("tt768_e4m3", 300, False),
                                            ("tt768_bf16", 1000, True),
                                            ("tt1024_4096_bf16", 4096, True)])
def test_noalloc_forward_matches_tt_forward(name, T, keep_z):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from tensor_train_compressed_tt_gb300 import _build, ttc
    _build.build()
    w = synth.WORKLOADS[name]
    s = w.layers[0]
    act = {"bf16": ttc.TT_DT_BF16, "f32": ttc.TT_DT_F32, "e4m3": ttc.TT_DT_E4M3}[w.act]
    ydt = torch.float32 if w.act == "f32" else torch.bfloat16
    inp = synth.draw(w, seed=7, tokens=T)
    # keep_z: the plan that also stores z' for a backward, which the no-alloc
    # call then writes into the library's array
    flags = ttc.TT_REUSE_Z if keep_z else 0
    plan = ttc.tt_plan(ttc.make_desc(s.in_modes, s.out_modes, s.ranks, act, flags))
    params = torch.from_numpy(synth.pack(inp.layers[0].cores, inp.layers[0].diags)).cuda()
    if w.act == "e4m3":
        x = torch.from_numpy(synth.e4m3_bytes(inp.x)).cuda()
    else:
        x = torch.from_numpy(inp.x).cuda().to(ydt)
    st = torch.cuda.current_stream().cuda_stream
    # the existing entry point with a caller-owned workspace
    ws = torch.empty(ttc.tt_workspace_size(plan, T), dtype=torch.uint8, device="cuda")
    y_ref = torch.empty((T, s.M), dtype=ydt, device="cuda")
    ttc.check(ttc.tt_forward(plan, T, x.data_ptr(), params.data_ptr(), y_ref.data_ptr(),
                             ws.data_ptr(), ws.numel(), st), "tt_forward")
    # two calls in a row through the C ABI, no workspace
    for _ in range(2):
        y = torch.full((T, s.M), float("nan"), dtype=ydt, device="cuda")
        ttc.check(ttc.tt_forward_noalloc(plan, T, x.data_ptr(), params.data_ptr(), y.data_ptr(),
                                         st), "tt_forward_noalloc")
        torch.cuda.synchronize()
        assert torch.isfinite(y.float()).all()
        assert torch.equal(y, y_ref)
    assert ttc.tt_get_device_status(st) == 0
