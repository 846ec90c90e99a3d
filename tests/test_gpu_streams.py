"""Calls that overlap on the GPU: two layers with multi-phase merge programs
(grid barriers between phases), each on its own stream with its own
workspace, launched back to back without synchronising.  Each program's
grid barrier counts arrivals in its own workspace, so the two cannot mix;
both results must match the oracle."""

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


from parity_util import TOL, compare, oracle_layer, to_dev  # noqa: E402


def test_two_streams_with_multi_phase_merges():
    from tensor_train_compressed_tt_gb300.layer import TTLinear
    jobs = []
    for name, T, seed in (("tt768_bf16", 1000, 71), ("tt1024_4096_bf16", 2048, 72),
                          ("tt768_bf16", 3000, 73), ("tt1024_4096_bf16", 700, 74)):
        w = synth.WORKLOADS[name]
        inp = synth.draw(w, seed=seed, tokens=T)
        sh = w.layers[0]
        lay = TTLinear(sh.in_modes, sh.out_modes, sh.ranks, torch.bfloat16)
        params = torch.from_numpy(synth.pack(inp.layers[0].cores, inp.layers[0].diags)).cuda()
        jobs.append(dict(sh=sh, inp=inp, lay=lay, params=params, x=to_dev(inp.x, "bf16"),
                         dy=to_dev(inp.dy, "bf16"), ws=lay.workspace(T),
                         stream=torch.cuda.Stream()))
    torch.cuda.synchronize()
    for rep in range(3):
        for j in jobs:   # every job's forward and backward queued before any sync
            with torch.cuda.stream(j["stream"]):
                j["y"] = j["lay"].forward(j["x"], j["params"], ws=j["ws"], stream=j["stream"])
                j["dx"], j["dp"] = j["lay"].backward(j["x"], j["dy"], j["params"], ws=j["ws"],
                                                     stream=j["stream"])
        torch.cuda.synchronize()
        for j in jobs:
            gc, gd = synth.unpack(j["sh"], j["dp"].cpu().numpy())
            out = {"y": j["y"].float().cpu().numpy(), "dx": j["dx"].float().cpu().numpy(),
                   "dcores": gc, "ddiags": gd}
            if rep == 0:
                j["ref"] = oracle_layer(j["sh"], j["inp"].layers[0], j["inp"].x, j["inp"].dy)
            compare(out, j["ref"], TOL["bf16"], f"{j['sh']} rep {rep}")
