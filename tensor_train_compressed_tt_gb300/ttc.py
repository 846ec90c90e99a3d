"""Thin ctypes binding of libttc (argument marshalling only).

Every function here forwards to the C entry point of the same name declared
in include/ttc.h; all arithmetic runs in the library's CUDA kernels.  The
binding raises if libttc.so has not been built: there is no other path.

Pointers are passed as integers (``tensor.data_ptr()``), streams as the
integer handle of a CUDA stream (``torch.cuda.current_stream().cuda_stream``).
"""

from __future__ import annotations

import ctypes
import os
from typing import List, Sequence, Tuple

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libttc.so")

TT_MAX_D = 4
TT_DT_F32 = 0
TT_DT_BF16 = 1
TT_DT_E4M3 = 2   # x, dy as one-byte FP8 E4M3 codes; y, dx bf16
TT_ACCUMULATE = 1
TT_REUSE_MERGE = 2
TT_REUSE_Z = 4   # forward keeps z' for the backward (implies TT_REUSE_MERGE)
TT_DETERMINISTIC = 8   # bit-reproducible gradients (fixed summation order)
TT_MULTI_MAX = 3       # layers of a multi-layer plan (one shared input)

STATUS = {
    0: "TT_OK",
    1: "TT_ERR_INVALID_ARG",
    2: "TT_ERR_UNSUPPORTED",
    3: "TT_ERR_WORKSPACE",
    4: "TT_ERR_CUDA",
    5: "TT_ERR_TIMEOUT",
    6: "TT_ERR_DEVICE",
}


class TTError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)}")


class tt_desc(ctypes.Structure):
    _fields_ = [
        ("d", ctypes.c_int),
        ("in_modes", ctypes.c_int * TT_MAX_D),
        ("out_modes", ctypes.c_int * TT_MAX_D),
        ("ranks", ctypes.c_int * (2 * TT_MAX_D + 1)),
        ("act", ctypes.c_int),
        ("flags", ctypes.c_uint),
    ]


class tt_ttm_desc(ctypes.Structure):
    _fields_ = [
        ("d", ctypes.c_int),
        ("row_modes", ctypes.c_int * TT_MAX_D),
        ("col_modes", ctypes.c_int * TT_MAX_D),
        ("ranks", ctypes.c_int * (TT_MAX_D + 1)),
        ("flags", ctypes.c_uint),
    ]


class tt_rank_opts(ctypes.Structure):
    _fields_ = [
        ("gamma", ctypes.c_float),
        ("beta", ctypes.c_float),
        ("lr", ctypes.c_float),
    ]


_lib = None
_P = ctypes.c_void_p
_SZ = ctypes.c_size_t
_I64 = ctypes.c_int64


def lib() -> ctypes.CDLL:
    """Load libttc.so once; raise loudly if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libttc.so not found at {LIB_PATH}; build it with "
                "`python -m tensor_train_compressed_tt_gb300._build`")
        L = ctypes.CDLL(LIB_PATH)
        sigs = {
            "tt_default_ranks": [ctypes.c_int, _P, _P, ctypes.c_int, _P],
            "tt_plan": [_P, _P],
            "tt_ffn_plan": [_P, _P, _P],
            "tt_destroy": [_P],
            "tt_param_layout": [_P, _P, _P, _P],
            "tt_ffn_param_layout": [_P, ctypes.c_int, _P, _P, _P],
            "tt_workspace_size": [_P, _I64, _P],
            "tt_forward": [_P, _I64, _P, _P, _P, _P, _SZ, _P],
            "tt_forward_noalloc": [_P, _I64, _P, _P, _P, _P],
            "tt_backward": [_P, _I64, _P, _P, _P, _P, _P, _P, _SZ, _P],
            "tt_ffn_forward": [_P, _I64, _P, _P, _P, _P, _P, _SZ, _P],
            "tt_ffn_backward": [_P, _I64, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P],
            "tt_multi_plan": [_P, ctypes.c_int, _P],
            "tt_multi_param_layout": [_P, ctypes.c_int, _P, _P, _P],
            "tt_multi_forward": [_P, _I64, _P, _P, _P, _P, _SZ, _P],
            "tt_multi_backward": [_P, _I64, _P, _P, _P, _P, _P, _SZ, _P],
            "tt_rank_update": [_P, _P, _P, _P, _P],
            "tt_backward_rank_update": [_P, _I64, _P, _P, _P, _P, _P, _P, _P, _SZ, _P],
            "tt_ttm_plan": [_P, _P],
            "tt_ttm_lookup": [_P, _I64, _P, _P, _P, _P, _SZ, _P],
            "tt_ttm_lookup_backward": [_P, _I64, _P, _P, _P, _P, _P, _SZ, _P],
            "tt_ttm_stats": [_P, _P, _P, _P, _P],
            "tt_get_device_status": [_P],
            "tt_set_wait_limit_ns": [ctypes.c_uint64],
            "tt_debug_skip_arrival": [ctypes.c_int],
            "tt_status_string": [ctypes.c_int],
        }
        for name, args in sigs.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        L.tt_destroy.restype = None
        L.tt_status_string.restype = ctypes.c_char_p
        L.tt_profile_enable.argtypes = [ctypes.c_int]
        L.tt_profile_enable.restype = None
        L.tt_profile_phase.argtypes = [ctypes.c_int, _P, _P]
        L.tt_profile_phase.restype = ctypes.c_int
        L.tt_profile_phase_name.argtypes = [ctypes.c_int]
        L.tt_profile_phase_name.restype = ctypes.c_char_p
        L.tt_launch_count.argtypes = []
        L.tt_launch_count.restype = ctypes.c_uint64
        L.tt_gelu_rate.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P]
        L.tt_gelu_rate.restype = ctypes.c_int
        _lib = L
    return _lib


def _check(code: int, where: str):
    if code != 0:
        raise TTError(code, where)


def make_desc(in_modes: Sequence[int], out_modes: Sequence[int], ranks: Sequence[int],
              act: int, flags: int = 0) -> tt_desc:
    d = len(in_modes)
    desc = tt_desc()
    desc.d = d
    for k in range(d):
        desc.in_modes[k] = int(in_modes[k])
        desc.out_modes[k] = int(out_modes[k])
    for k, r in enumerate(ranks):
        desc.ranks[k] = int(r)
    desc.act = int(act)
    desc.flags = int(flags)
    return desc


def tt_default_ranks(in_modes: Sequence[int], out_modes: Sequence[int], R: int) -> List[int]:
    d = len(in_modes)
    a = (ctypes.c_int * d)(*in_modes)
    b = (ctypes.c_int * d)(*out_modes)
    out = (ctypes.c_int * (2 * d + 1))()
    _check(lib().tt_default_ranks(d, a, b, int(R), out), "tt_default_ranks")
    return list(out)


class Plan:
    """Owns one tt_plan_t handle (single layer or FFN pair)."""

    def __init__(self, handle: int, kind: str, d: Tuple[int, ...]):
        self.handle = handle
        self.kind = kind
        self.d = d

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.tt_destroy(ctypes.c_void_p(self.handle))
            self.handle = None


def tt_plan(desc: tt_desc) -> Plan:
    h = ctypes.c_void_p()
    _check(lib().tt_plan(ctypes.byref(desc), ctypes.byref(h)), "tt_plan")
    return Plan(h.value, "linear", (desc.d,))


def tt_ffn_plan(up: tt_desc, down: tt_desc) -> Plan:
    h = ctypes.c_void_p()
    _check(lib().tt_ffn_plan(ctypes.byref(up), ctypes.byref(down), ctypes.byref(h)),
           "tt_ffn_plan")
    return Plan(h.value, "ffn", (up.d, down.d))


def tt_multi_plan(descs: Sequence[tt_desc]) -> Plan:
    arr = (tt_desc * len(descs))(*descs)
    h = ctypes.c_void_p()
    _check(lib().tt_multi_plan(arr, len(descs), ctypes.byref(h)), "tt_multi_plan")
    return Plan(h.value, "multi", tuple(d.d for d in descs))


def _layout(fn, args, d):
    core = (ctypes.c_size_t * (2 * d))()
    diag = (ctypes.c_size_t * max(1, 2 * d - 1))()
    n = ctypes.c_size_t()
    _check(fn(*args, core, diag, ctypes.byref(n)), fn.__name__)
    return list(core), list(diag)[: 2 * d - 1], n.value


def tt_param_layout(plan: Plan):
    core, diag, n = _layout(lib().tt_param_layout, [ctypes.c_void_p(plan.handle)], plan.d[0])
    if plan.kind == "ttm":  # a TT-matrix table: d cores, d-1 diagonals
        d = plan.d[0]
        return core[:d], diag[:d - 1], n
    return core, diag, n


def tt_ffn_param_layout(plan: Plan, layer: int):
    return _layout(lib().tt_ffn_param_layout, [ctypes.c_void_p(plan.handle), int(layer)],
                   plan.d[layer])


def tt_multi_param_layout(plan: Plan, layer: int):
    d = plan.d[layer] if 0 <= layer < len(plan.d) else plan.d[0]   # the library checks layer
    return _layout(lib().tt_multi_param_layout, [ctypes.c_void_p(plan.handle), int(layer)], d)


def tt_workspace_size(plan: Plan, T: int) -> int:
    n = ctypes.c_size_t()
    _check(lib().tt_workspace_size(ctypes.c_void_p(plan.handle), int(T), ctypes.byref(n)),
           "tt_workspace_size")
    return n.value


def tt_forward(plan: Plan, T: int, x: int, params: int, y: int, ws: int, ws_bytes: int,
               stream: int = 0) -> int:
    """Returns the tt_status code (0 = TT_OK)."""
    return lib().tt_forward(ctypes.c_void_p(plan.handle), int(T), x, params, y, ws,
                            int(ws_bytes), stream)


def tt_forward_noalloc(plan: Plan, T: int, x: int, params: int, y: int, stream: int = 0) -> int:
    """tt_forward with the library's fixed device scratch (no caller workspace)."""
    return lib().tt_forward_noalloc(ctypes.c_void_p(plan.handle), int(T), x, params, y, stream)


def tt_backward(plan: Plan, T: int, x: int, dy: int, params: int, dx: int, dparams: int,
                ws: int, ws_bytes: int, stream: int = 0) -> int:
    return lib().tt_backward(ctypes.c_void_p(plan.handle), int(T), x, dy, params, dx, dparams,
                             ws, int(ws_bytes), stream)


def tt_ffn_forward(plan: Plan, T: int, x: int, params_up: int, params_down: int, y: int,
                   ws: int, ws_bytes: int, stream: int = 0) -> int:
    return lib().tt_ffn_forward(ctypes.c_void_p(plan.handle), int(T), x, params_up,
                                params_down, y, ws, int(ws_bytes), stream)


def tt_ffn_backward(plan: Plan, T: int, x: int, dy: int, params_up: int, params_down: int,
                    dx: int, dparams_up: int, dparams_down: int, ws: int, ws_bytes: int,
                    stream: int = 0) -> int:
    return lib().tt_ffn_backward(ctypes.c_void_p(plan.handle), int(T), x, dy, params_up,
                                 params_down, dx, dparams_up, dparams_down, ws,
                                 int(ws_bytes), stream)


def _ptrs(ps: Sequence[int]):
    return (ctypes.c_void_p * len(ps))(*[ctypes.c_void_p(int(p)) for p in ps])


def tt_multi_forward(plan: Plan, T: int, x: int, params: Sequence[int], y: Sequence[int],
                     ws: int, ws_bytes: int, stream: int = 0) -> int:
    """params, y: one device pointer a layer (host arrays built here)."""
    return lib().tt_multi_forward(ctypes.c_void_p(plan.handle), int(T), x, _ptrs(params),
                                  _ptrs(y), ws, int(ws_bytes), stream)


def tt_multi_backward(plan: Plan, T: int, x: int, dy: Sequence[int], params: Sequence[int],
                      dx: int, dparams: Sequence[int], ws: int, ws_bytes: int,
                      stream: int = 0) -> int:
    """dx receives the sum over the layers of dy_g W_g."""
    return lib().tt_multi_backward(ctypes.c_void_p(plan.handle), int(T), x, _ptrs(dy),
                                   _ptrs(params), dx, _ptrs(dparams), ws, int(ws_bytes),
                                   stream)


def tt_rank_update(plan: Plan, params: int, dparams: int, gamma: float, beta: float,
                   lr: float, stream: int = 0) -> int:
    """Penalty sub-gradient (lr == 0) or proximal step (lr > 0), in place."""
    o = tt_rank_opts(float(gamma), float(beta), float(lr))
    return lib().tt_rank_update(ctypes.c_void_p(plan.handle), params, dparams,
                                ctypes.byref(o), stream)


def tt_backward_rank_update(plan: Plan, T: int, x: int, dy: int, params: int, dx: int,
                            dparams: int, gamma: float, beta: float, lr: float, ws: int,
                            ws_bytes: int, stream: int = 0) -> int:
    """tt_backward then the rank-adaptive step, the step inside the merge program."""
    o = tt_rank_opts(float(gamma), float(beta), float(lr))
    return lib().tt_backward_rank_update(ctypes.c_void_p(plan.handle), int(T), x, dy, params, dx,
                                         dparams, ctypes.byref(o), ws, int(ws_bytes), stream)


def make_ttm_desc(row_modes: Sequence[int], col_modes: Sequence[int], ranks: Sequence[int],
                  flags: int = 0) -> tt_ttm_desc:
    desc = tt_ttm_desc()
    desc.d = len(row_modes)
    for k in range(len(row_modes)):
        desc.row_modes[k] = int(row_modes[k])
        desc.col_modes[k] = int(col_modes[k])
    for k, r in enumerate(ranks):
        desc.ranks[k] = int(r)
    desc.flags = int(flags)
    return desc


def tt_ttm_plan(desc: tt_ttm_desc) -> Plan:
    h = ctypes.c_void_p()
    _check(lib().tt_ttm_plan(ctypes.byref(desc), ctypes.byref(h)), "tt_ttm_plan")
    return Plan(h.value, "ttm", (desc.d,))


def tt_ttm_lookup(plan: Plan, B: int, idx: int, params: int, out: int, ws: int, ws_bytes: int,
                  stream: int = 0) -> int:
    return lib().tt_ttm_lookup(ctypes.c_void_p(plan.handle), int(B), idx, params, out, ws,
                               int(ws_bytes), stream)


def tt_ttm_lookup_backward(plan: Plan, B: int, idx: int, dout: int, params: int, dparams: int,
                           ws: int, ws_bytes: int, stream: int = 0) -> int:
    return lib().tt_ttm_lookup_backward(ctypes.c_void_p(plan.handle), int(B), idx, dout, params,
                                        dparams, ws, int(ws_bytes), stream)


def tt_ttm_stats(plan: Plan, ws: int, stream: int = 0):
    u = ctypes.c_int64()
    p = ctypes.c_int64()
    _check(lib().tt_ttm_stats(ctypes.c_void_p(plan.handle), ws, ctypes.byref(u),
                              ctypes.byref(p), stream), "tt_ttm_stats")
    return u.value, p.value


def tt_get_device_status(stream: int = 0) -> int:
    return lib().tt_get_device_status(stream)


TT_DEBUG_NONE = 0
TT_DEBUG_FWD_TOKENS = 1
TT_DEBUG_BWD_TOKENS = 2
TT_DEBUG_MERGE_BARRIER = 3


def tt_set_wait_limit_ns(ns: int) -> int:
    """Limit of the kernels' bounded waits on the current device (ns)."""
    return lib().tt_set_wait_limit_ns(int(ns))


def tt_debug_skip_arrival(site: int) -> int:
    """Test hook: the next launch of `site` skips one arrival in its first CTA."""
    return lib().tt_debug_skip_arrival(int(site))


def tt_status_string(code: int) -> str:
    return lib().tt_status_string(int(code)).decode()


def check(code: int, where: str = "libttc"):
    """Raise TTError for a non-zero status code."""
    _check(code, where)
