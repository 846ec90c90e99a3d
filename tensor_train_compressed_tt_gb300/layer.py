"""PyTorch-facing wrappers over the libttc C ABI.

PyTorch supplies device memory and the stream; each method marshals tensor
pointers into one libttc call.  No arithmetic happens here.
"""

from __future__ import annotations

from typing import Optional, Sequence

import torch

from . import ttc

_DT = {torch.float32: ttc.TT_DT_F32, torch.bfloat16: ttc.TT_DT_BF16}
# E4M3 activations: x / dy hold one-byte codes (a float8_e4m3fn tensor, or
# uint8 holding the same bytes); y / dx come back in bf16.
if hasattr(torch, "float8_e4m3fn"):
    _DT[torch.float8_e4m3fn] = ttc.TT_DT_E4M3
_DT[torch.uint8] = ttc.TT_DT_E4M3


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> int:
    return 0 if t is None else int(t.data_ptr())


class TTLinear:
    """One TT linear layer: y (T x M) = x (T x N) W^T, W given by packed cores."""

    def __init__(self, in_modes: Sequence[int], out_modes: Sequence[int],
                 ranks: Sequence[int], dtype: torch.dtype = torch.bfloat16,
                 accumulate: bool = False, reuse_merge: bool = False, reuse_z: bool = False,
                 deterministic: bool = False):
        self.in_modes = tuple(in_modes)
        self.out_modes = tuple(out_modes)
        self.ranks = tuple(ranks)
        self.dtype = dtype
        # dtype of y and dx
        self.out_dtype = torch.bfloat16 if _DT[dtype] == ttc.TT_DT_E4M3 else dtype
        flags = (ttc.TT_ACCUMULATE if accumulate else 0) | \
            (ttc.TT_REUSE_MERGE if reuse_merge else 0) | (ttc.TT_REUSE_Z if reuse_z else 0) | \
            (ttc.TT_DETERMINISTIC if deterministic else 0)
        self.desc = ttc.make_desc(in_modes, out_modes, ranks, _DT[dtype], flags)
        self.plan = ttc.tt_plan(self.desc)
        self.core_off, self.diag_off, self.n_params = ttc.tt_param_layout(self.plan)
        self.N = 1
        self.M = 1
        for n in in_modes:
            self.N *= n
        for m in out_modes:
            self.M *= m

    def workspace_bytes(self, T: int) -> int:
        return ttc.tt_workspace_size(self.plan, T)

    def workspace(self, T: int, device="cuda") -> torch.Tensor:
        return torch.empty(self.workspace_bytes(T), dtype=torch.uint8, device=device)

    def forward(self, x: torch.Tensor, params: torch.Tensor, y: Optional[torch.Tensor] = None,
                ws: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        T = x.shape[0]
        if y is None:
            y = torch.empty((T, self.M), dtype=self.out_dtype, device=x.device)
        if ws is None:
            ws = self.workspace(T, x.device)
        ttc.check(ttc.tt_forward(self.plan, T, _ptr(x), _ptr(params), _ptr(y), _ptr(ws),
                                 ws.numel(), _stream(stream)), "tt_forward")
        return y

    def backward(self, x: torch.Tensor, dy: torch.Tensor, params: torch.Tensor,
                 dx: Optional[torch.Tensor] = None, dparams: Optional[torch.Tensor] = None,
                 ws: Optional[torch.Tensor] = None, stream=None):
        T = x.shape[0]
        if dx is None:
            dx = torch.empty((T, self.N), dtype=self.out_dtype, device=x.device)
        if dparams is None:
            dparams = torch.empty(self.n_params, dtype=torch.float32, device=x.device)
        if ws is None:
            ws = self.workspace(T, x.device)
        ttc.check(ttc.tt_backward(self.plan, T, _ptr(x), _ptr(dy), _ptr(params), _ptr(dx),
                                  _ptr(dparams), _ptr(ws), ws.numel(), _stream(stream)),
                  "tt_backward")
        return dx, dparams


    def rank_update(self, params: torch.Tensor, dparams: torch.Tensor, gamma: float,
                    beta: float, lr: float = 0.0, stream=None) -> None:
        """In place: dparams += penalty sub-gradient (lr == 0), or one
        proximal gradient step on params (lr > 0)."""
        ttc.check(ttc.tt_rank_update(self.plan, _ptr(params), _ptr(dparams), gamma, beta, lr,
                                     _stream(stream)), "tt_rank_update")


class TTFFN:
    """y = TT_down(GELU(TT_up(x))), exact erf GELU, both layers through one plan."""

    def __init__(self, up: Sequence[Sequence[int]], down: Sequence[Sequence[int]],
                 dtype: torch.dtype = torch.bfloat16, accumulate: bool = False,
                 reuse_merge: bool = False, reuse_z: bool = False, deterministic: bool = False):
        flags = (ttc.TT_ACCUMULATE if accumulate else 0) | \
            (ttc.TT_REUSE_MERGE if reuse_merge else 0) | (ttc.TT_REUSE_Z if reuse_z else 0) | \
            (ttc.TT_DETERMINISTIC if deterministic else 0)
        self.dtype = dtype
        self.up_desc = ttc.make_desc(up[0], up[1], up[2], _DT[dtype], flags)
        self.down_desc = ttc.make_desc(down[0], down[1], down[2], _DT[dtype], flags)
        self.plan = ttc.tt_ffn_plan(self.up_desc, self.down_desc)
        self.layout = [ttc.tt_ffn_param_layout(self.plan, i) for i in (0, 1)]
        self.N = 1
        self.M = 1
        for n in up[0]:
            self.N *= n
        for m in down[1]:
            self.M *= m

    def workspace(self, T: int, device="cuda") -> torch.Tensor:
        return torch.empty(ttc.tt_workspace_size(self.plan, T), dtype=torch.uint8,
                           device=device)

    def forward(self, x, p_up, p_down, y=None, ws=None, stream=None):
        T = x.shape[0]
        if y is None:
            y = torch.empty((T, self.M), dtype=self.dtype, device=x.device)
        if ws is None:
            ws = self.workspace(T, x.device)
        ttc.check(ttc.tt_ffn_forward(self.plan, T, _ptr(x), _ptr(p_up), _ptr(p_down), _ptr(y),
                                     _ptr(ws), ws.numel(), _stream(stream)), "tt_ffn_forward")
        return y

    def backward(self, x, dy, p_up, p_down, dx=None, dp_up=None, dp_down=None, ws=None,
                 stream=None):
        T = x.shape[0]
        if dx is None:
            dx = torch.empty((T, self.N), dtype=self.dtype, device=x.device)
        if dp_up is None:
            dp_up = torch.empty(self.layout[0][2], dtype=torch.float32, device=x.device)
        if dp_down is None:
            dp_down = torch.empty(self.layout[1][2], dtype=torch.float32, device=x.device)
        if ws is None:
            ws = self.workspace(T, x.device)
        ttc.check(ttc.tt_ffn_backward(self.plan, T, _ptr(x), _ptr(dy), _ptr(p_up),
                                      _ptr(p_down), _ptr(dx), _ptr(dp_up), _ptr(dp_down),
                                      _ptr(ws), ws.numel(), _stream(stream)),
                  "tt_ffn_backward")
        return dx, dp_up, dp_down


class TTMulti:
    """Up to three TT layers on one input x (the Q, K and V projections):
    y_g = x W_g^T for each layer; the backward returns dx = sum_g dy_g W_g
    and each layer's packed gradients."""

    def __init__(self, layers: Sequence[Sequence[Sequence[int]]],
                 dtype: torch.dtype = torch.bfloat16, accumulate: bool = False,
                 reuse_merge: bool = False, reuse_z: bool = False, deterministic: bool = False):
        flags = (ttc.TT_ACCUMULATE if accumulate else 0) | \
            (ttc.TT_REUSE_MERGE if reuse_merge else 0) | (ttc.TT_REUSE_Z if reuse_z else 0) | \
            (ttc.TT_DETERMINISTIC if deterministic else 0)
        self.dtype = dtype
        self.out_dtype = torch.bfloat16 if _DT[dtype] == ttc.TT_DT_E4M3 else dtype
        self.descs = [ttc.make_desc(i, o, r, _DT[dtype], flags) for i, o, r in layers]
        self.plan = ttc.tt_multi_plan(self.descs)
        self.G = len(self.descs)
        self.layout = [ttc.tt_multi_param_layout(self.plan, g) for g in range(self.G)]
        self.N = 1
        for n in layers[0][0]:
            self.N *= n
        self.M = []
        for _, o, _ in layers:
            m = 1
            for v in o:
                m *= v
            self.M.append(m)

    def workspace(self, T: int, device="cuda") -> torch.Tensor:
        return torch.empty(ttc.tt_workspace_size(self.plan, T), dtype=torch.uint8,
                           device=device)

    def forward(self, x, params, y=None, ws=None, stream=None):
        T = x.shape[0]
        if y is None:
            y = [torch.empty((T, m), dtype=self.out_dtype, device=x.device) for m in self.M]
        if ws is None:
            ws = self.workspace(T, x.device)
        ttc.check(ttc.tt_multi_forward(self.plan, T, _ptr(x), [_ptr(p) for p in params],
                                       [_ptr(t) for t in y], _ptr(ws), ws.numel(),
                                       _stream(stream)), "tt_multi_forward")
        return y

    def backward(self, x, dy, params, dx=None, dparams=None, ws=None, stream=None):
        T = x.shape[0]
        if dx is None:
            dx = torch.empty((T, self.N), dtype=self.out_dtype, device=x.device)
        if dparams is None:
            dparams = [torch.empty(lay[2], dtype=torch.float32, device=x.device)
                       for lay in self.layout]
        if ws is None:
            ws = self.workspace(T, x.device)
        ttc.check(ttc.tt_multi_backward(self.plan, T, _ptr(x), [_ptr(t) for t in dy],
                                        [_ptr(p) for p in params], _ptr(dx),
                                        [_ptr(t) for t in dparams], _ptr(ws), ws.numel(),
                                        _stream(stream)), "tt_multi_backward")
        return dx, dparams


class TTMEmbedding:
    """TT-matrix embedding table: lookup of rows for int32 indices and its
    backward into the packed cores/diagonals (float32)."""

    def __init__(self, row_modes: Sequence[int], col_modes: Sequence[int],
                 ranks: Sequence[int], accumulate: bool = False, reuse: bool = False):
        # reuse: backward() takes the batch's distinct rows from the lookup()
        # of the same indices on the same workspace (TT_REUSE_MERGE)
        flags = (ttc.TT_ACCUMULATE if accumulate else 0) | (ttc.TT_REUSE_MERGE if reuse else 0)
        self.desc = ttc.make_ttm_desc(row_modes, col_modes, ranks, flags)
        self.plan = ttc.tt_ttm_plan(self.desc)
        self.core_off, self.diag_off, self.n_params = ttc.tt_param_layout(self.plan)
        self.V = 1
        self.Dm = 1
        for m in row_modes:
            self.V *= m
        for n in col_modes:
            self.Dm *= n

    def workspace(self, B: int, device="cuda") -> torch.Tensor:
        return torch.empty(ttc.tt_workspace_size(self.plan, B), dtype=torch.uint8, device=device)

    def lookup(self, idx: torch.Tensor, params: torch.Tensor, out=None, ws=None, stream=None):
        B = idx.shape[0]
        if out is None:
            out = torch.empty((B, self.Dm), dtype=torch.float32, device=idx.device)
        if ws is None:
            ws = self.workspace(B, idx.device)
        ttc.check(ttc.tt_ttm_lookup(self.plan, B, _ptr(idx), _ptr(params), _ptr(out), _ptr(ws),
                                    ws.numel(), _stream(stream)), "tt_ttm_lookup")
        return out

    def backward(self, idx: torch.Tensor, dout: torch.Tensor, params: torch.Tensor,
                 dparams=None, ws=None, stream=None):
        B = idx.shape[0]
        if dparams is None:
            dparams = torch.empty(self.n_params, dtype=torch.float32, device=idx.device)
        if ws is None:
            ws = self.workspace(B, idx.device)
        ttc.check(ttc.tt_ttm_lookup_backward(self.plan, B, _ptr(idx), _ptr(dout), _ptr(params),
                                             _ptr(dparams), _ptr(ws), ws.numel(),
                                             _stream(stream)), "tt_ttm_lookup_backward")
        return dparams

    def stats(self, ws: torch.Tensor, stream=None):
        """(distinct rows, distinct (i_1, i_2) prefixes) of the last call on ws."""
        return ttc.tt_ttm_stats(self.plan, _ptr(ws), _stream(stream))
