"""Shared helpers of the GPU parity tests: run libttc and the oracle on the
same seeded inputs and compare every output tensor."""

from __future__ import annotations

import numpy as np
import torch

from oracle import tt_oracle as O
from tensor_train_compressed_tt_gb300 import synth
from tensor_train_compressed_tt_gb300.layer import TTFFN, TTLinear

# E4M3 inputs: the products run on bf16 tiles (the E4M3 values widened
# exactly) with bf16 merged operands and bf16 outputs, so the bf16 bound holds.
TOL = {"f32": 1e-4, "bf16": 2e-2, "e4m3": 2e-2}
TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16, "e4m3": torch.uint8}


def to_dev(a: np.ndarray, act: str) -> torch.Tensor:
    if act == "e4m3":   # one-byte codes of values that are E4M3-representable
        return torch.from_numpy(synth.e4m3_bytes(a)).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda().to(TORCH_DT[act])


def gpu_layer(shape: synth.LayerShape, act: str, li: synth.LayerInputs, x: np.ndarray,
              dy: np.ndarray, accumulate: bool = False, reuse_z: bool = False):
    """Forward then backward on one workspace (reuse_z: the backward reads the
    forward's kept z', as the benchmark's step does)."""
    layer = TTLinear(shape.in_modes, shape.out_modes, shape.ranks, TORCH_DT[act], accumulate,
                     reuse_z=reuse_z)
    params = torch.from_numpy(synth.pack(li.cores, li.diags)).cuda()
    xd, dyd = to_dev(x, act), to_dev(dy, act)
    T = x.shape[0]
    ws = layer.workspace(T)
    y = layer.forward(xd, params, ws=ws)
    dx, dp = layer.backward(xd, dyd, params, ws=ws)
    torch.cuda.synchronize()
    cores, diags = synth.unpack(shape, dp.cpu().numpy())
    return {"y": y.float().cpu().numpy(), "dx": dx.float().cpu().numpy(),
            "dcores": cores, "ddiags": diags}


def oracle_layer(shape: synth.LayerShape, li: synth.LayerInputs, x, dy):
    cores = [c.astype(np.float64) for c in li.cores]
    diags = [e.astype(np.float64) for e in li.diags]
    y = O.chained_forward(cores, diags, shape.d, x)
    dx, dC, dE = O.chained_backward(cores, diags, shape.d, x, dy, prune_convention=True)
    return {"y": y, "dx": dx, "dcores": dC, "ddiags": dE}


def compare(out, ref, tol, label=""):
    """Norm-wise relative error per tensor; exact zeros where the reference is zero."""
    errs = {}

    def one(name, a, b):
        e = O.rel_err(a, b)
        errs[name] = e
        assert e <= tol, f"{label} {name}: rel err {e:.3e} > {tol:.1e}"
        zero = np.asarray(b) == 0.0
        if np.any(zero):
            assert np.all(np.asarray(a)[zero] == 0.0), f"{label} {name}: nonzero where ref is 0"

    one("y", out["y"], ref["y"])
    one("dx", out["dx"], ref["dx"])
    for k, (a, b) in enumerate(zip(out["dcores"], ref["dcores"])):
        one(f"dG{k + 1}", a, b)
    for k, (a, b) in enumerate(zip(out["ddiags"], ref["ddiags"])):
        one(f"dD{k + 1}", a, b)
    return errs


def gpu_ffn(w: synth.Workload, inp: synth.WorkloadInputs, reuse_z: bool = False):
    """Forward then backward on one workspace (reuse_z: the backward takes the
    forward's merges, z', h and GELU(h), as the benchmark's step does)."""
    up, dn = w.layers
    ffn = TTFFN((up.in_modes, up.out_modes, up.ranks), (dn.in_modes, dn.out_modes, dn.ranks),
                TORCH_DT[w.act], reuse_z=reuse_z)
    pu = torch.from_numpy(synth.pack(inp.layers[0].cores, inp.layers[0].diags)).cuda()
    pd = torch.from_numpy(synth.pack(inp.layers[1].cores, inp.layers[1].diags)).cuda()
    xd, dyd = to_dev(inp.x, w.act), to_dev(inp.dy, w.act)
    ws = ffn.workspace(inp.x.shape[0])
    y = ffn.forward(xd, pu, pd, ws=ws)
    dx, dpu, dpd = ffn.backward(xd, dyd, pu, pd, ws=ws)
    torch.cuda.synchronize()
    cu, du = synth.unpack(up, dpu.cpu().numpy())
    cd, dd = synth.unpack(dn, dpd.cpu().numpy())
    return ({"y": y.float().cpu().numpy(), "dx": dx.float().cpu().numpy()},
            (cu, du), (cd, dd))


def oracle_ffn(w: synth.Workload, inp: synth.WorkloadInputs):
    up, dn = w.layers
    pu = ([c.astype(np.float64) for c in inp.layers[0].cores],
          [e.astype(np.float64) for e in inp.layers[0].diags])
    pd = ([c.astype(np.float64) for c in inp.layers[1].cores],
          [e.astype(np.float64) for e in inp.layers[1].diags])
    y = O.ffn_forward(pu, pd, up.d, dn.d, inp.x)
    dx, gu, gd = O.ffn_backward(pu, pd, up.d, dn.d, inp.x, inp.dy, prune_convention=True)
    return {"y": y, "dx": dx}, gu, gd
