"""Multi-rank paths on CPU (gloo, world size 2).

The benchmark's bookkeeping: each rank runs its own replica; the step time is
the slowest rank's and the value counts the tokens of every rank.  And the
one exchange a data-parallel training step needs: the token sums behind
dparams are linear in the tokens, so one all-reduce (sum) of the replicas'
packed dparams gives the gradient of the whole batch.
"""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.all_reduce_scalar(1.5 + rank, "max")
    k = bench.all_reduce_scalar(100 - 7 * rank, "min")
    tot = bench.all_reduce_scalar(rank + 1, "sum")
    rate = bench.whole_job_rate(16384, world, ms)
    q.put((rank, ms, k, tot, rate))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_like_the_benchmark():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, k, tot, rate in res:
        assert ms == 2.5 and k == 93 and tot == 3
        assert rate == pytest.approx(2 * 16384 / 2.5e-3)


def _grad_worker(rank, world, port, q):
    """Rank r takes rows r::world of one seeded batch, runs the oracle's
    backward on them, all-reduces its packed dparams (and reassembles dx by
    all-gather) over gloo."""
    import numpy as np
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from oracle import tt_oracle as O
    from tensor_train_compressed_tt_gb300 import synth
    w = synth.WORKLOADS["tiny64_f32"]
    inp = synth.draw(w, seed=7, tokens=24)
    sh = w.layers[0]
    li = inp.layers[0]
    cores = [c.astype(np.float64) for c in li.cores]
    diags = [e.astype(np.float64) for e in li.diags]
    xs, dys = inp.x[rank::world], inp.dy[rank::world]
    dx, dC, dE = O.chained_backward(cores, diags, sh.d, xs, dys)
    flat = torch.from_numpy(synth.pack([c.astype(np.float32) for c in dC],
                                       [e.astype(np.float32) for e in dE]).astype(np.float64))
    dist.all_reduce(flat, op=dist.ReduceOp.SUM)
    parts = [torch.zeros(dx.shape, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(parts, torch.from_numpy(np.ascontiguousarray(dx)))
    q.put((rank, flat.numpy(), [p.numpy() for p in parts]))
    dist.barrier()
    dist.destroy_process_group()


def test_all_reduced_dparams_equal_the_whole_batch_gradient():
    import numpy as np
    from oracle import tt_oracle as O
    from tensor_train_compressed_tt_gb300 import synth
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_grad_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=120) for _ in range(world)), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w = synth.WORKLOADS["tiny64_f32"]
    inp = synth.draw(w, seed=7, tokens=24)
    sh, li = w.layers[0], inp.layers[0]
    cores = [c.astype(np.float64) for c in li.cores]
    diags = [e.astype(np.float64) for e in li.diags]
    dx, dC, dE = O.chained_backward(cores, diags, sh.d, inp.x, inp.dy)
    whole = synth.pack([c.astype(np.float32) for c in dC], [e.astype(np.float32) for e in dE])
    for rank, flat, parts in res:
        # the float32 packing of each half rounds once more than the whole's
        assert O.rel_err(flat, whole) <= 1e-6
        dx_all = np.empty_like(dx)
        for r, part in enumerate(parts):
            dx_all[r::world] = part
        assert O.rel_err(dx_all, dx) <= 1e-12
    assert np.array_equal(res[0][1], res[1][1])


def test_single_process_is_identity():
    import bench
    assert bench.all_reduce_scalar(3.25, "max") == 3.25
    assert bench.whole_job_rate(100, 1, 1.0) == pytest.approx(1e5)


def test_graph_steps_are_whole_passes_over_the_sets():
    """A graph replay runs whole passes over the rotating input sets (every
    set as often as the others), several passes for a few sets, one pass once
    the sets alone reach the 64-step limit."""
    import bench
    for nsets in (2, 3, 4, 16, 17, 64, 65, 16545):
        for passes in (1, 2, 4):
            g = bench.graph_steps(nsets, passes)
            assert g % nsets == 0 and nsets <= g <= nsets * passes
            assert g <= max(64, nsets)
    assert bench.graph_steps(4, 4) == 16
    assert bench.graph_steps(16545, 4) == 16545
    assert bench.graph_steps(4, 0) == 4


def test_algorithmic_bytes_per_activation_type():
    """The roofline's algorithmic bytes: x read by both passes, dy read, y and
    dx written, at the bytes of an input element (E4M3: 1) and of an output
    element (bf16: 2)."""
    import bench
    from tensor_train_compressed_tt_gb300 import synth
    T, N, M = 16384, 768, 768
    bf = bench.algorithmic(synth.WORKLOADS["tt768_bf16"], T)
    f8 = bench.algorithmic(synth.WORKLOADS["tt768_e4m3"], T)
    assert bf["bytes"] == 2 * T * (3 * N + 2 * M)
    assert bf["fwd_bytes"] == 2 * T * (N + M) and bf["bwd_bytes"] == 2 * T * (2 * N + M)
    assert f8["bytes"] == T * (2 * N + M + 2 * (M + N))
    assert f8["fwd_bytes"] == T * (N + 2 * M) and f8["bwd_bytes"] == T * (N + M + 2 * N)
    r = 30
    assert bf["flop"] == f8["flop"] == 6 * T * r * (N + M)
