"""Host-side checks of the libttc C ABI (no GPU work is launched here)."""

import ctypes
import os
import re

import numpy as np
import pytest

from oracle import tt_oracle as O
from tensor_train_compressed_tt_gb300 import synth, ttc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from tensor_train_compressed_tt_gb300 import _build
    _build.build()
    return ttc.lib()


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        txt = open(os.path.join(ROOT, "include", fn)).read()
        txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
        names |= set(re.findall(r"\b(tt_[a-z_0-9]+)\s*\(", txt))
    return names


def test_library_exports_every_declared_symbol(lib):
    names = _declared_symbols()
    assert {"tt_plan", "tt_forward", "tt_backward", "tt_workspace_size"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), n


def _desc(shape, act=ttc.TT_DT_BF16, flags=0):
    return ttc.make_desc(shape.in_modes, shape.out_modes, shape.ranks, act, flags)


def test_default_ranks_match_oracle(lib):
    rng = np.random.default_rng(3)
    for _ in range(50):
        d = int(rng.integers(1, 5))
        im = [int(v) for v in rng.integers(1, 20, size=d)]
        om = [int(v) for v in rng.integers(1, 20, size=d)]
        R = int(rng.integers(1, 80))
        assert ttc.tt_default_ranks(im, om, R) == O.rank_caps(im, om, R)


@pytest.mark.parametrize("name", sorted(synth.WORKLOADS))
def test_param_layout_matches_pack(lib, name):
    w = synth.WORKLOADS[name]
    for shape in w.layers:
        plan = ttc.tt_plan(_desc(shape))
        core_off, diag_off, n = ttc.tt_param_layout(plan)
        off = 0
        for k, cs in enumerate(shape.core_shapes()):
            assert core_off[k] == off
            off += int(np.prod(cs))
        for e, ds in enumerate(shape.diag_sizes()):
            assert diag_off[e] == off
            off += ds
        assert n == off


def test_ffn_layout_and_validation(lib):
    w = synth.WORKLOADS["ffn768_3072_bf16"]
    up, dn = w.layers
    plan = ttc.tt_ffn_plan(_desc(up), _desc(dn))
    for i, shape in enumerate((up, dn)):
        _, _, n = ttc.tt_ffn_param_layout(plan, i)
        assert n == sum(int(np.prod(c)) for c in shape.core_shapes()) + sum(shape.diag_sizes())
    with pytest.raises(ttc.TTError):
        ttc.tt_ffn_plan(_desc(up), _desc(up))   # widths do not chain
    with pytest.raises(ttc.TTError):
        ttc.tt_ffn_plan(_desc(up), _desc(dn, act=ttc.TT_DT_F32))


def test_reuse_z_flag(lib):
    """TT_REUSE_Z adds T x 64 bf16 of kept z' to the tensor-core plans'
    workspace, implies TT_REUSE_MERGE, and leaves f32 plans alone."""
    shape = synth.WORKLOADS["tt768_bf16"].layers[0]
    for act in (ttc.TT_DT_BF16, ttc.TT_DT_E4M3):
        base = ttc.tt_plan(_desc(shape, act=act))
        kz = ttc.tt_plan(_desc(shape, act=act, flags=ttc.TT_REUSE_Z))
        km = ttc.tt_plan(_desc(shape, act=act, flags=ttc.TT_REUSE_Z | ttc.TT_REUSE_MERGE))
        for T in (1, 300, 16384):
            extra = ttc.tt_workspace_size(kz, T) - ttc.tt_workspace_size(base, T)
            assert T * 128 <= extra < T * 128 + 512
            assert ttc.tt_workspace_size(km, T) == ttc.tt_workspace_size(kz, T)
    f32 = ttc.tt_plan(_desc(shape, act=ttc.TT_DT_F32))
    f32z = ttc.tt_plan(_desc(shape, act=ttc.TT_DT_F32, flags=ttc.TT_REUSE_Z))
    assert ttc.tt_workspace_size(f32z, 1000) == ttc.tt_workspace_size(f32, 1000)
    # FFN (fused bf16 pair): each layer always has a region of its own and its
    # z' (T x 64 bf16), which the backward reads; no T x hidden buffers
    up, dn = synth.WORKLOADS["ffn768_3072_bf16"].layers
    a = ttc.tt_ffn_plan(_desc(up), _desc(dn))
    b = ttc.tt_ffn_plan(_desc(up, flags=ttc.TT_REUSE_Z), _desc(dn, flags=ttc.TT_REUSE_Z))
    for T in (1, 4096, 16384):
        assert ttc.tt_workspace_size(b, T) == ttc.tt_workspace_size(a, T)
        assert 2 * T * 128 <= ttc.tt_workspace_size(a, T) - ttc.tt_workspace_size(a, 0) \
            < 2 * T * 128 + 2048
    assert ttc.tt_workspace_size(a, 16384) < 16384 * up.M * 2   # h never stored
    with pytest.raises(ttc.TTError):   # the two layers must carry the same flags
        ttc.tt_ffn_plan(_desc(up, flags=ttc.TT_REUSE_Z), _desc(dn))


def test_multi_plan_layout_and_validation(lib):
    """A multi-layer plan takes 1..3 layers with the same input modes, act
    type and flags; each layer keeps its own packed layout.  The fused bf16
    plan holds one region a layer with its z' (T x 64 bf16); the
    layer-by-layer plans (f32, TT_DETERMINISTIC) hold the other layers' dx
    instead."""
    L = synth.ENCODER_LAYERS
    q, up = L["q"], L["up"]
    plan = ttc.tt_multi_plan([_desc(q), _desc(q), _desc(up)])
    for g, shape in enumerate((q, q, up)):
        core_off, diag_off, n = ttc.tt_multi_param_layout(plan, g)
        assert n == sum(int(np.prod(c)) for c in shape.core_shapes()) + sum(shape.diag_sizes())
        assert core_off[0] == 0 and diag_off[0] == n - sum(shape.diag_sizes())
    with pytest.raises(ttc.TTError):
        ttc.tt_multi_param_layout(plan, 3)
    with pytest.raises(ttc.TTError):
        ttc.tt_multi_plan([])
    with pytest.raises(ttc.TTError):
        ttc.tt_multi_plan([_desc(q)] * 4)
    with pytest.raises(ttc.TTError):   # input modes differ
        ttc.tt_multi_plan([_desc(q), _desc(L["down"])])
    with pytest.raises(ttc.TTError):   # act types differ
        ttc.tt_multi_plan([_desc(q), _desc(q, act=ttc.TT_DT_F32)])
    with pytest.raises(ttc.TTError):   # flags differ
        ttc.tt_multi_plan([_desc(q), _desc(q, flags=ttc.TT_REUSE_Z)])
    one = ttc.tt_plan(_desc(q))
    fused = ttc.tt_multi_plan([_desc(q)] * 3)
    for T in (1, 1000, 16384):
        w1 = ttc.tt_workspace_size(one, T)
        w3 = ttc.tt_workspace_size(fused, T)
        assert 3 * (w1 + T * 128) <= w3 + 3 * 512 and w3 <= 3 * (w1 + T * 128) + 3 * 512
    # the layer-by-layer backward (f32) keeps the dx of layers 2 and 3 before
    # the sum; the fused bf16 kernels, deterministic or not, sum dx on the SM
    def extra(act, flags, T):
        single = ttc.tt_plan(_desc(q, act=act, flags=flags))
        multi = ttc.tt_multi_plan([_desc(q, act=act, flags=flags)] * 3)
        return ttc.tt_workspace_size(multi, T) - 3 * ttc.tt_workspace_size(single, T)

    for T in (7, 1000):
        e = extra(ttc.TT_DT_F32, 0, T)
        assert 2 * T * q.N * 4 - 3 * 512 <= e <= 2 * T * q.N * 4 + 3 * 512
        assert extra(ttc.TT_DT_BF16, ttc.TT_DETERMINISTIC, T) == extra(ttc.TT_DT_BF16, 0, T)
    assert extra(ttc.TT_DT_BF16, ttc.TT_DETERMINISTIC, 1000) < 2 * 1000 * q.N * 2


def test_multi_argument_errors_return_before_any_launch(lib):
    q = synth.ENCODER_LAYERS["q"]
    plan = ttc.tt_multi_plan([_desc(q)] * 3)
    need = ttc.tt_workspace_size(plan, 64)
    fake = 1 << 40
    p3 = [fake] * 3
    assert ttc.tt_multi_forward(plan, 0, 0, p3, [0] * 3, 0, 0) == 0      # T == 0: no-op
    assert ttc.tt_multi_forward(plan, -1, fake, p3, p3, fake, need) == 1
    assert ttc.tt_multi_forward(plan, 64, fake, [fake, 0, fake], p3, fake, need) == 1
    assert ttc.tt_multi_forward(plan, 64, fake, p3, [fake, fake + 2, fake], fake, need) == 1
    assert ttc.tt_multi_forward(plan, 64, fake, p3, p3, fake, need - 1) == 3
    assert ttc.tt_multi_backward(plan, 64, fake, p3, p3, fake, [fake, fake, 0], fake, need) == 1
    assert ttc.tt_multi_backward(plan, 64, fake, [fake, fake + 8, fake], p3, fake, p3, fake,
                                 need) == 1
    assert ttc.tt_multi_backward(plan, 64, fake, p3, p3, fake + 4, p3, fake, need) == 1
    assert ttc.tt_multi_backward(plan, 64, fake, p3, p3, fake, p3, fake + 16, need) == 3
    single = ttc.tt_plan(_desc(q))   # a single-layer plan is not a multi plan
    assert ttc.tt_multi_forward(single, 64, fake, p3, p3, fake, need) == 1
    assert ttc.tt_forward(plan, 64, fake, fake, fake, fake, need) == 1


def test_deterministic_flag_workspace(lib):
    """TT_DETERMINISTIC adds one token-sum slot per CTA of the backward
    (128-token tiles, at most 160) to the tensor-core plans' workspace."""
    shape = synth.WORKLOADS["tt768_bf16"].layers[0]
    base = ttc.tt_plan(_desc(shape))
    det = ttc.tt_plan(_desc(shape, flags=ttc.TT_DETERMINISTIC))
    slot = (shape.N + shape.M + 4) * 64 * 4
    for T, slots in ((1, 1), (300, 3), (16384, 128), (10 ** 6, 160)):
        extra = ttc.tt_workspace_size(det, T) - ttc.tt_workspace_size(base, T)
        assert slots * slot <= extra < slots * slot + 512
    f32 = ttc.tt_plan(_desc(shape, act=ttc.TT_DT_F32, flags=ttc.TT_DETERMINISTIC))
    assert ttc.tt_workspace_size(f32, 999) == ttc.tt_workspace_size(
        ttc.tt_plan(_desc(shape, act=ttc.TT_DT_F32)), 999)


def test_e4m3_plans(lib):
    """E4M3 runs on the fused tensor-core kernels only: shapes they do not
    take, and FFN pairs, are refused at plan time; the workspace is the bf16
    plan's (no f32 token scratch)."""
    shape = synth.WORKLOADS["tt768_e4m3"].layers[0]
    plan = ttc.tt_plan(_desc(shape, act=ttc.TT_DT_E4M3))
    bf = ttc.tt_plan(_desc(shape))
    for T in (0, 1, 16384):
        assert ttc.tt_workspace_size(plan, T) == ttc.tt_workspace_size(bf, T)
    bad = [synth.LayerShape((12, 8, 9), (8, 8, 12), (1, 12, 30, 30, 30, 12, 1)),  # N = 864 ok
           synth.LayerShape((8, 17, 1), (8, 8, 12), (1, 8, 30, 30, 30, 12, 1)),   # N = 136
           synth.LayerShape((4, 4, 4), (4, 4, 4), (1, 4, 8, 8, 8, 4, 1)),           # N < 128
           synth.LayerShape((16, 16), (16, 16), (1, 16, 72, 16, 1))]                # r_d > 64
    ttc.tt_plan(_desc(bad[0], act=ttc.TT_DT_E4M3))
    for b in bad[1:]:
        with pytest.raises(ttc.TTError) as e:
            ttc.tt_plan(_desc(b, act=ttc.TT_DT_E4M3))
        assert e.value.code == 2
        ttc.tt_plan(_desc(b))   # the bf16 plan of the same shape is fine
    up, dn = synth.WORKLOADS["ffn768_3072_bf16"].layers
    with pytest.raises(ttc.TTError) as e:
        ttc.tt_ffn_plan(_desc(up, act=ttc.TT_DT_E4M3), _desc(dn, act=ttc.TT_DT_E4M3))
    assert e.value.code == 2


@pytest.mark.parametrize("mutate", [
    lambda d: setattr(d, "d", 0),
    lambda d: setattr(d, "d", 5),
    lambda d: d.ranks.__setitem__(0, 2),
    lambda d: d.ranks.__setitem__(6, 3),
    lambda d: d.ranks.__setitem__(3, 0),
    lambda d: d.in_modes.__setitem__(1, 0),
    lambda d: setattr(d, "act", 7),
    lambda d: setattr(d, "flags", 0x80),
    lambda d: setattr(d, "flags", 0x10),
])
def test_invalid_descriptors_rejected(lib, mutate):
    shape = synth.WORKLOADS["tt768_bf16"].layers[0]
    desc = _desc(shape)
    mutate(desc)
    with pytest.raises(ttc.TTError) as e:
        ttc.tt_plan(desc)
    assert e.value.code == 1


def test_workspace_size_grows_with_tokens(lib):
    plan = ttc.tt_plan(_desc(synth.WORKLOADS["tt768_bf16"].layers[0]))
    a = ttc.tt_workspace_size(plan, 0)
    b = ttc.tt_workspace_size(plan, 128)
    c = ttc.tt_workspace_size(plan, 16384)
    assert 0 < a <= b <= c and a % 256 == 0 and c % 256 == 0


def test_argument_errors_return_before_any_launch(lib):
    plan = ttc.tt_plan(_desc(synth.WORKLOADS["tt768_bf16"].layers[0]))
    ws_need = ttc.tt_workspace_size(plan, 64)
    fake = 1 << 40   # never dereferenced: every call below fails its host checks
    # T == 0 is a no-op for the forward
    assert ttc.tt_forward(plan, 0, 0, 0, 0, 0, 0) == 0
    assert ttc.tt_forward(plan, -1, fake, fake, fake, fake, ws_need) == 1
    assert ttc.tt_forward(plan, 64, 0, fake, fake, fake, ws_need) == 1          # NULL x
    assert ttc.tt_forward(plan, 64, fake + 2, fake, fake, fake, ws_need) == 1   # misaligned x
    assert ttc.tt_forward(plan, 64, fake, fake, fake, 0, ws_need) == 3          # no workspace
    assert ttc.tt_forward(plan, 64, fake, fake, fake, fake + 16, ws_need) == 3  # misaligned ws
    assert ttc.tt_forward(plan, 64, fake, fake, fake, fake, ws_need - 1) == 3   # too small
    assert ttc.tt_backward(plan, 64, fake, fake, fake, fake, 0, fake, ws_need) == 1
    assert ttc.tt_backward(plan, 64, fake, fake + 8, fake, fake, fake, fake, ws_need) == 1
    # a single-layer plan is not an FFN plan
    assert ttc.tt_ffn_forward(plan, 64, fake, fake, fake, fake, fake, ws_need) == 1
    # rank step: null buffers, negative or non-finite weights, FFN plans
    assert ttc.tt_rank_update(plan, 0, fake, 0.1, 0.1, 0.1) == 1
    assert ttc.tt_rank_update(plan, fake, 0, 0.1, 0.1, 0.1) == 1
    assert ttc.tt_rank_update(plan, fake, fake, -0.1, 0.1, 0.1) == 1
    assert ttc.tt_rank_update(plan, fake, fake, 0.1, -0.1, 0.1) == 1
    assert ttc.tt_rank_update(plan, fake, fake, 0.1, 0.1, -0.1) == 1
    assert ttc.tt_rank_update(plan, fake, fake, float("nan"), 0.1, 0.1) == 1
    assert ttc.tt_rank_update(plan, fake, fake, 0.1, float("inf"), 0.1) == 1
    w = synth.WORKLOADS["ffn768_3072_bf16"]
    ffn = ttc.tt_ffn_plan(_desc(w.layers[0]), _desc(w.layers[1]))
    assert ttc.tt_rank_update(ffn, fake, fake, 0.1, 0.1, 0.1) == 1
    # backward with the fused step: the step's weights and the plan kind first
    assert ttc.tt_backward_rank_update(plan, 64, fake, fake, fake, fake, fake, -1.0, 0.1, 0.1,
                                       fake, ws_need) == 1
    assert ttc.tt_backward_rank_update(plan, 64, fake, fake, fake, fake, fake, 0.1, float("nan"),
                                       0.1, fake, ws_need) == 1
    assert ttc.tt_backward_rank_update(ffn, 64, fake, fake, fake, fake, fake, 0.1, 0.1, 0.1,
                                       fake, ws_need) == 1
    assert ttc.tt_backward_rank_update(plan, 64, fake, fake, fake, fake, fake, 0.1, 0.1, 0.1,
                                       fake, ws_need - 1) == 3


def test_noalloc_rejections_before_any_launch(lib):
    """tt_forward_noalloc checks everything on the host first: a layer whose
    scratch would exceed the library's fixed 32 MiB array gets
    TT_ERR_WORKSPACE, an FFN plan or T < 0 TT_ERR_INVALID_ARG, T == 0 is a
    no-op; none of these touches a device."""
    limit = 32 << 20
    fake = 1 << 40
    shape = synth.WORKLOADS["tt1024_4096_bf16"].layers[0]
    for act, flags in ((ttc.TT_DT_BF16, ttc.TT_REUSE_Z), (ttc.TT_DT_F32, 0)):
        plan = ttc.tt_plan(_desc(shape, act=act, flags=flags))
        T = 1024
        while ttc.tt_workspace_size(plan, T) <= limit:
            T *= 2
        assert ttc.tt_forward_noalloc(plan, T, fake, fake, fake) == 3
        assert ttc.tt_workspace_size(plan, 257) <= limit
    plan = ttc.tt_plan(_desc(shape))
    assert ttc.tt_forward_noalloc(plan, 0, 0, 0, 0) == 0
    assert ttc.tt_forward_noalloc(plan, -1, fake, fake, fake) == 1
    w = synth.WORKLOADS["ffn768_3072_bf16"]
    ffn = ttc.tt_ffn_plan(_desc(w.layers[0]), _desc(w.layers[1]))
    assert ttc.tt_forward_noalloc(ffn, 64, fake, fake, fake) == 1
    table = ttc.tt_ttm_plan(ttc.make_ttm_desc((32, 32, 32), (8, 8, 12), (1, 30, 30, 1)))
    assert ttc.tt_forward_noalloc(table, 64, fake, fake, fake) == 1


def test_ttm_plan_and_argument_errors(lib):
    plan = ttc.tt_ttm_plan(ttc.make_ttm_desc((32, 32, 32), (8, 8, 12), (1, 30, 30, 1)))
    core, diag, n = ttc.tt_param_layout(plan)
    t = synth.draw_ttm(synth.TTM_WORKLOADS["ttm_emb_10k"], batch=4)
    assert n == synth.pack(t.cores, t.diags).size
    assert core == [0, 7680, 238080] and diag == [249600, 249630]
    a = ttc.tt_workspace_size(plan, 10000)
    b = ttc.tt_workspace_size(plan, 40000)
    assert 0 < a < b
    for bad in [((32,), (8,), (1, 1)),                       # d = 1
                ((32, 32, 32), (8, 8, 12), (2, 30, 30, 1)),  # r_0 != 1
                ((32, 0, 32), (8, 8, 12), (1, 30, 30, 1))]:  # empty mode
        with pytest.raises(ttc.TTError) as e:
            ttc.tt_ttm_plan(ttc.make_ttm_desc(*bad))
        assert e.value.code == 1
    with pytest.raises(ttc.TTError) as e:   # rank above 64: no kernel
        ttc.tt_ttm_plan(ttc.make_ttm_desc((32, 32), (8, 8), (1, 65, 1)))
    assert e.value.code == 2
    # TT_ACCUMULATE and TT_REUSE_MERGE are a TTM plan's flags; TT_REUSE_Z is not
    flags = ttc.TT_ACCUMULATE | ttc.TT_REUSE_MERGE
    ttc.tt_ttm_plan(ttc.make_ttm_desc((32, 32, 32), (8, 8, 12), (1, 30, 30, 1), flags))
    with pytest.raises(ttc.TTError) as e:
        ttc.tt_ttm_plan(ttc.make_ttm_desc((32, 32, 32), (8, 8, 12), (1, 30, 30, 1),
                                          ttc.TT_REUSE_Z))
    assert e.value.code == 1
    fake = 1 << 40
    ws = ttc.tt_workspace_size(plan, 64)
    assert ttc.tt_ttm_lookup(plan, 0, 0, 0, 0, 0, 0) == 0                    # B == 0
    assert ttc.tt_ttm_lookup(plan, -1, fake, fake, fake, fake, ws) == 1
    assert ttc.tt_ttm_lookup(plan, 64, 0, fake, fake, fake, ws) == 1         # NULL idx
    assert ttc.tt_ttm_lookup(plan, 64, fake, fake, fake + 4, fake, ws) == 1  # misaligned out
    assert ttc.tt_ttm_lookup(plan, 64, fake, fake, fake, fake, ws - 1) == 3  # small workspace
    assert ttc.tt_ttm_lookup(plan, 64, fake, fake, fake, fake + 64, ws) == 3 # misaligned ws
    assert ttc.tt_ttm_lookup_backward(plan, 64, fake, fake, 0, fake, fake, ws) == 1
    # a TT-layer plan is not a table and the reverse
    layer = ttc.tt_plan(_desc(synth.WORKLOADS["tt768_bf16"].layers[0]))
    assert ttc.tt_ttm_lookup(layer, 64, fake, fake, fake, fake, ws) == 1
    assert ttc.tt_forward(plan, 64, fake, fake, fake, fake, ws) == 1
    assert ttc.tt_rank_update(plan, fake, fake, 0.1, 0.1, 0.1) == 1


def test_status_strings(lib):
    for code, name in ttc.STATUS.items():
        assert ttc.tt_status_string(code).startswith(name)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """No CPU fallback: without libttc.so the binding raises instead of
    computing anything."""
    monkeypatch.setattr(ttc, "LIB_PATH", str(tmp_path / "absent" / "libttc.so"))
    monkeypatch.setattr(ttc, "_lib", None)   # both restored after the test
    with pytest.raises(RuntimeError, match="not found"):
        ttc.lib()
