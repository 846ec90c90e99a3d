"""The TT layers of one transformer encoder block as one step.

The CoMERA project page tensorises every linear layer of its encoder blocks
(the attention projections Q, K, V, O and the feed-forward pair) and runs the
whole training step as one CUDA graph to remove launch overhead ("Making small
tensor operations fast on GPUs", bullet "CUDA Graph": 14.3 -> 7.2 minutes an
epoch).  This module composes the library's calls for one block: the forward
of Q, K, V (on the same x: one multi-layer plan, whose kernels stream x once
for all three), O and the FFN pair, then their backward in reverse order, all
on one stream so that a CUDA graph captures the block with the
programmatic-launch edges between consecutive kernels.  The backward of Q, K
and V returns their summed input gradient dx_q + dx_k + dx_v, which is what
the block's x receives.  The attention between
the projections is not a TT layer and is not part of this step.

Argument marshalling only: every product runs in libttc's kernels.
"""

from __future__ import annotations

from typing import Dict

import torch

from . import synth, ttc
from .layer import TTFFN, TTLinear, TTMulti

PROJ = ("q", "k", "v", "o")
QKV = ("q", "k", "v")


class TTEncoderBlock:
    """Q, K, V, O (768 x 768) and the GELU FFN pair (768 -> 3072 -> 768), each
    a rank-30 TT layer, bf16 activations; the backward of every layer reuses
    its forward's merges and kept z' (TT_REUSE_Z)."""

    def __init__(self, reuse_z: bool = True, deterministic: bool = False,
                 fuse_qkv: bool = True):
        L = synth.ENCODER_LAYERS
        self.fuse_qkv = fuse_qkv
        single = ("o",) if fuse_qkv else PROJ
        self.proj = {nm: TTLinear(L[nm].in_modes, L[nm].out_modes, L[nm].ranks, torch.bfloat16,
                                  reuse_z=reuse_z, deterministic=deterministic) for nm in single}
        self.qkv = TTMulti([(L[nm].in_modes, L[nm].out_modes, L[nm].ranks) for nm in QKV],
                           torch.bfloat16, reuse_z=reuse_z,
                           deterministic=deterministic) if fuse_qkv else None
        up, dn = L["up"], L["down"]
        self.ffn = TTFFN((up.in_modes, up.out_modes, up.ranks),
                         (dn.in_modes, dn.out_modes, dn.ranks), torch.bfloat16,
                         reuse_z=reuse_z, deterministic=deterministic)

    def buffers(self, T: int, device="cuda") -> Dict[str, torch.Tensor]:
        """Workspaces, outputs and gradients of one step (allocated once)."""
        b = {}
        if self.fuse_qkv:
            b["ws_qkv"] = self.qkv.workspace(T, device)
            b["dx_qkv"] = torch.empty((T, self.qkv.N), dtype=torch.bfloat16, device=device)
            for g, nm in enumerate(QKV):
                b[f"y_{nm}"] = torch.empty((T, self.qkv.M[g]), dtype=torch.bfloat16,
                                           device=device)
                b[f"dp_{nm}"] = torch.empty(self.qkv.layout[g][2], dtype=torch.float32,
                                            device=device)
        for nm in self.proj:
            lay = self.proj[nm]
            b[f"ws_{nm}"] = lay.workspace(T, device)
            b[f"y_{nm}"] = torch.empty((T, lay.M), dtype=torch.bfloat16, device=device)
            b[f"dx_{nm}"] = torch.empty((T, lay.N), dtype=torch.bfloat16, device=device)
            b[f"dp_{nm}"] = torch.empty(lay.n_params, dtype=torch.float32, device=device)
        b["ws_ffn"] = self.ffn.workspace(T, device)
        b["y_ffn"] = torch.empty((T, self.ffn.M), dtype=torch.bfloat16, device=device)
        b["dx_ffn"] = torch.empty((T, self.ffn.N), dtype=torch.bfloat16, device=device)
        b["dp_up"] = torch.empty(self.ffn.layout[0][2], dtype=torch.float32, device=device)
        b["dp_down"] = torch.empty(self.ffn.layout[1][2], dtype=torch.float32, device=device)
        return b

    def step(self, x, xo, xf, dy: Dict[str, torch.Tensor], params: Dict[str, torch.Tensor],
             b: Dict[str, torch.Tensor], stream=None) -> None:
        """Forward of Q, K, V, O and the FFN pair, then the backward in reverse
        order; outputs in b (y_* and dp_* per layer, dx_* per input: dx_qkv
        for the fused Q, K, V)."""
        xin = {"q": x, "k": x, "v": x, "o": xo}
        if self.fuse_qkv:
            self.qkv.forward(x, [params[nm] for nm in QKV], y=[b[f"y_{nm}"] for nm in QKV],
                             ws=b["ws_qkv"], stream=stream)
        for nm in self.proj:
            self.proj[nm].forward(xin[nm], params[nm], y=b[f"y_{nm}"], ws=b[f"ws_{nm}"],
                                  stream=stream)
        self.ffn.forward(xf, params["up"], params["down"], y=b["y_ffn"], ws=b["ws_ffn"],
                         stream=stream)
        self.ffn.backward(xf, dy["ffn"], params["up"], params["down"], dx=b["dx_ffn"],
                          dp_up=b["dp_up"], dp_down=b["dp_down"], ws=b["ws_ffn"], stream=stream)
        for nm in reversed(list(self.proj)):
            self.proj[nm].backward(xin[nm], dy[nm], params[nm], dx=b[f"dx_{nm}"],
                                   dparams=b[f"dp_{nm}"], ws=b[f"ws_{nm}"], stream=stream)
        if self.fuse_qkv:
            self.qkv.backward(x, [dy[nm] for nm in QKV], [params[nm] for nm in QKV],
                              dx=b["dx_qkv"], dparams=[b[f"dp_{nm}"] for nm in QKV],
                              ws=b["ws_qkv"], stream=stream)

    def capture(self, T, x, xo, xf, dy, params, b) -> torch.cuda.CUDAGraph:
        """The step as one CUDA graph (replay() runs the whole block)."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step(x, xo, xf, dy, params, b)  # on the capture stream
        return g
