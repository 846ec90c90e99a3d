"""GPU parity of the TT-matrix embedding lookup (tt_ttm_lookup and its
backward) against the fp64 oracle.

The lookup is fp32 arithmetic (short sums over ranks), so rows and gradients
must match the oracle within the fp32 tolerance (1e-4 norm-wise); the
de-duplication is integer work and must match exactly (distinct rows and
distinct (i_1, i_2) prefixes of the batch).
"""

import numpy as np
import pytest

from oracle import tt_oracle as O
from tensor_train_compressed_tt_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from tensor_train_compressed_tt_gb300 import _build
    _build.build()


def _run(shape, cores, diags, idx, dout, accumulate=False, base=None, reuse=False):
    from tensor_train_compressed_tt_gb300.layer import TTMEmbedding
    emb = TTMEmbedding(shape.row_modes, shape.col_modes, shape.ranks, accumulate=accumulate,
                       reuse=reuse)
    p = torch.from_numpy(synth.pack(cores, diags)).cuda()
    i = torch.from_numpy(np.asarray(idx, np.int32)).cuda()
    g = torch.from_numpy(np.asarray(dout, np.float32)).cuda()
    ws = emb.workspace(len(idx))
    out = emb.lookup(i, p, ws=ws)
    stats_f = emb.stats(ws)
    dp = torch.from_numpy(base.copy()).cuda() if base is not None else None
    dp = emb.backward(i, g, p, dparams=dp, ws=ws)
    stats_b = emb.stats(ws)
    from tensor_train_compressed_tt_gb300 import ttc
    ttc.check(ttc.tt_get_device_status(0), "device status")
    return out.cpu().numpy(), dp.cpu().numpy(), stats_f, stats_b


def _check(shape, cores, diags, idx, dout, label, reuse=False):
    out, dp, sf, sb = _run(shape, cores, diags, idx, dout, reuse=reuse)
    c64 = [c.astype(np.float64) for c in cores]
    d64 = [e.astype(np.float64) for e in diags]
    ref = O.ttm_lookup(c64, d64, idx)
    assert O.rel_err(out, ref) <= TOL, label
    dC, dE = O.ttm_lookup_backward(c64, d64, idx, dout)
    gc, gd = synth_unpack(shape, dp)
    for k, (a, b) in enumerate(zip(gc, dC)):
        assert O.rel_err(a, b) <= TOL, f"{label} dF_{k + 1}"
    for k, (a, b) in enumerate(zip(gd, dE)):
        assert O.rel_err(a, b) <= TOL, f"{label} dD_{k + 1}"
        assert np.all(a[np.asarray(diags[k]) == 0] == 0)
    m = shape.row_modes
    uniq = np.unique(idx)
    pairs = np.unique(uniq // (m[2] if len(m) == 3 else 1))
    assert sf == (uniq.size, pairs.size) and sb == sf, label


def synth_unpack(shape, flat):
    cores, diags, off = [], [], 0
    for cs in shape.core_shapes():
        n = int(np.prod(cs))
        cores.append(flat[off:off + n].reshape(cs))
        off += n
    for n in shape.diag_sizes():
        diags.append(flat[off:off + n])
        off += n
    assert off == flat.size
    return cores, diags


@pytest.mark.parametrize("m,n,r", [((4, 3, 5), (2, 3, 4), (1, 3, 5, 1)),
                                   ((6, 7), (4, 5), (1, 6, 1)),
                                   ((2, 2, 2), (1, 1, 1), (1, 1, 1, 1)),
                                   ((8, 4, 8), (4, 4, 6), (1, 16, 12, 1))])
def test_small_tables(m, n, r):
    rng = np.random.Generator(np.random.PCG64(41))
    shape = synth.TtmShape(m, n, r)
    cores = [(rng.standard_normal(cs) * 0.5).astype(np.float32) for cs in shape.core_shapes()]
    diags = [rng.uniform(0.5, 1.5, k).astype(np.float32) for k in shape.diag_sizes()]
    if diags and diags[0].size > 1:
        diags[0][0] = 0.0   # a pruned rank
    for B in (1, 37, 500):
        idx = rng.integers(0, shape.V, B).astype(np.int32)
        idx[: B // 3] = idx[0]   # repeated rows
        dout = rng.standard_normal((B, shape.Dm)).astype(np.float32)
        _check(shape, cores, diags, idx, dout, f"{m}x{n} r{r} B={B}")


@pytest.mark.parametrize("name,reuse", [("ttm_emb_10k", False), ("ttm_emb_40k", False),
                                        ("ttm_emb_40k", True)])
def test_workloads(name, reuse):
    """reuse: the backward takes the lookup's distinct rows and prefixes from
    the workspace (TT_REUSE_MERGE), as the benchmark's step runs it."""
    w = synth.TTM_WORKLOADS[name]
    t = synth.draw_ttm(w)
    _check(w.shape, t.cores, t.diags, t.idx, t.dout, name, reuse=reuse)


def test_reused_bookkeeping_twice_in_a_row():
    """Two backward calls after one lookup under TT_REUSE_MERGE give the same
    gradients as a backward that finds the distinct rows itself."""
    from tensor_train_compressed_tt_gb300.layer import TTMEmbedding
    w = synth.TTM_WORKLOADS["ttm_emb_10k"]
    t = synth.draw_ttm(w, seed=9, batch=3000)
    S = w.shape
    p = torch.from_numpy(synth.pack(t.cores, t.diags)).cuda()
    i = torch.from_numpy(t.idx).cuda()
    g = torch.from_numpy(t.dout).cuda()
    plain = TTMEmbedding(S.row_modes, S.col_modes, S.ranks)
    ref = plain.backward(i, g, p, ws=plain.workspace(3000))
    emb = TTMEmbedding(S.row_modes, S.col_modes, S.ranks, reuse=True)
    ws = emb.workspace(3000)
    emb.lookup(i, p, ws=ws)
    for _ in range(2):
        dp = emb.backward(i, g, p, ws=ws)
        torch.cuda.synchronize()
        assert O.rel_err(dp.cpu().numpy(), ref.cpu().numpy()) <= 1e-5


def test_accumulate_adds_into_dparams():
    w = synth.TTM_WORKLOADS["ttm_emb_10k"]
    t = synth.draw_ttm(w, batch=2000)
    _, g1, _, _ = _run(w.shape, t.cores, t.diags, t.idx, t.dout)
    base = np.full(g1.size, 0.5, np.float32)
    _, g2, _, _ = _run(w.shape, t.cores, t.diags, t.idx, t.dout, accumulate=True, base=base)
    assert O.rel_err(g2 - base, g1) <= 1e-5


def test_zero_batch_and_bad_index():
    from tensor_train_compressed_tt_gb300 import ttc
    from tensor_train_compressed_tt_gb300.layer import TTMEmbedding
    w = synth.TTM_WORKLOADS["ttm_emb_10k"]
    t = synth.draw_ttm(w, batch=64)
    emb = TTMEmbedding(w.shape.row_modes, w.shape.col_modes, w.shape.ranks)
    p = torch.from_numpy(synth.pack(t.cores, t.diags)).cuda()
    # B == 0: the backward writes zero gradients
    dp = torch.full((emb.n_params,), 3.0, device="cuda")
    ws = emb.workspace(1)
    ttc.check(ttc.tt_ttm_lookup_backward(emb.plan, 0, 0, 0, p.data_ptr(), dp.data_ptr(),
                                         ws.data_ptr(), ws.numel(), 0))
    torch.cuda.synchronize()
    assert torch.count_nonzero(dp).item() == 0
    # an index outside the table is skipped and reported; the others are looked up
    idx = torch.from_numpy(t.idx.copy()).cuda()
    idx[5] = w.shape.V + 7
    out = torch.full((64, w.shape.Dm), -1.0, device="cuda")
    emb.lookup(idx, p, out=out)
    assert ttc.tt_get_device_status(0) == 6   # TT_ERR_DEVICE
    assert ttc.tt_get_device_status(0) == 0   # read and cleared
    o = out.cpu().numpy()
    assert np.all(o[5] == -1.0)
    keep = np.arange(64) != 5
    ref = O.ttm_lookup([c.astype(np.float64) for c in t.cores],
                       [e.astype(np.float64) for e in t.diags], t.idx[keep])
    assert O.rel_err(o[keep], ref) <= TOL
