"""tt_forward_noalloc: the forward for callers that cannot allocate device memory.

Such callers (a plain-C host or plugin without a device allocator, or a
process that must not call cudaMalloc once running) get the scratch from a
fixed device array inside the library instead of a caller workspace.  This
file is collected last on purpose, so that a failure here cannot hide the
result of any other test; it must also pass when run on its own.
"""

import numpy as np
import pytest

from tensor_train_compressed_tt_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.mark.parametrize("name,T,tol", [("tt768_bf16", 300, 2e-2), ("tiny64_f32", 16, 1e-4),
                                         ("tt1024_4096_bf16", 257, 2e-2)])
def test_noalloc_forward_matches_tt_forward(name, T, tol):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from tensor_train_compressed_tt_gb300 import _build, ttc
    _build.build()
    w = synth.WORKLOADS[name]
    s = w.layers[0]
    dt = torch.bfloat16 if w.act == "bf16" else torch.float32
    inp = synth.draw(w, seed=7, tokens=T)
    plan = ttc.tt_plan(ttc.make_desc(s.in_modes, s.out_modes, s.ranks,
                                     ttc.TT_DT_BF16 if w.act == "bf16" else ttc.TT_DT_F32))
    params = torch.from_numpy(synth.pack(inp.layers[0].cores, inp.layers[0].diags)).cuda()
    x = torch.from_numpy(inp.x).cuda().to(dt)
    st = torch.cuda.current_stream().cuda_stream
    # the existing entry point with a caller-owned workspace
    ws = torch.empty(ttc.tt_workspace_size(plan, T), dtype=torch.uint8, device="cuda")
    y_ref = torch.empty((T, s.M), dtype=dt, device="cuda")
    ttc.check(ttc.tt_forward(plan, T, x.data_ptr(), params.data_ptr(), y_ref.data_ptr(),
                             ws.data_ptr(), ws.numel(), st), "tt_forward")
    ref = y_ref.float().cpu().numpy()
    # two calls in a row through the C ABI, no workspace
    for _ in range(2):
        y = torch.full((T, s.M), float("nan"), dtype=dt, device="cuda")
        ttc.check(ttc.tt_forward_noalloc(plan, T, x.data_ptr(), params.data_ptr(), y.data_ptr(),
                                         st), "tt_forward_noalloc")
        torch.cuda.synchronize()
        out = y.float().cpu().numpy()
        err = np.linalg.norm(out - ref) / np.linalg.norm(ref)
        assert np.isfinite(out).all() and err <= tol, err
    assert ttc.tt_get_device_status(st) == 0
