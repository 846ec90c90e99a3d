#!/usr/bin/env python3
"""Benchmark of the TT-linear forward + backward on one GB300 (or N replicas).

A step is one pass of the whole hot path over one batch of synthetic input:
tt_forward then tt_backward of the 768x768 TT layer (modes (12,8,8)x(8,8,12),
ranks 30, 16384 tokens, bf16 activations) by default.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on the host cores

Under torchrun every rank runs its own replica (tokens are independent rows;
no data-path collective); the timing is the max over ranks and the value is
the tokens of all ranks over that time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "TT-linear fwd+bwd tokens/s on 1 GB300 and % of roofline; CPU-oracle speedup"
DEFAULT_WORKLOAD = "tt768_bf16"
ELEM = {"bf16": 2, "f32": 4, "e4m3": 1}   # bytes of an x / dy element
OUT_ELEM = {"bf16": 2, "f32": 4, "e4m3": 2}   # bytes of a y / dx element (E4M3 in, bf16 out)


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--tokens", type=int, default=None)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--graph-passes", type=int, default=4,
                   help="passes over the rotating input sets one CUDA graph holds "
                        "(fewer where that would pass 64 steps a replay)")
    p.add_argument("--eager", action="store_true",
                   help="launch every step from the host instead of replaying a CUDA graph")
    p.add_argument("--no-reuse", action="store_true",
                   help="re-merge the cores in the backward instead of reusing the forward's")
    p.add_argument("--no-reuse-z", action="store_true",
                   help="recompute z' = x A diag(D) in the backward instead of keeping the forward's")
    p.add_argument("--no-fuse-qkv", action="store_true",
                   help="encoder block: Q, K and V as three single-layer plans")
    p.add_argument("--deterministic", action="store_true",
                   help="TT_DETERMINISTIC: fixed-order (bit-reproducible) gradient sums")
    p.add_argument("--oracle-rate", action="store_true", help=argparse.SUPPRESS)
    p.add_argument("--target-seconds", type=float, default=1.5,
                   help="the K-step timed region is repeated until the repeats last this "
                        "long (and at least 50 times)")
    return p.parse_args()


# ---------------------------------------------------------------------------
# shared helpers


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def algorithmic(w, T):
    """FLOP and bytes of one fwd+bwd step, and bytes per token pass of each kernel.

    FLOP = 6 T r' (N + M) per layer (the merged contraction order: x A, z' B,
    dy B^T, z'^T dy, dz A^T, x^T dz); bytes = T (2N ei + M ei + M eo + N eo)
    per layer (x read by both passes, dy read, y and dx written), ei / eo the
    bytes of an input / output element (bf16: 2 / 2, E4M3 in, bf16 out: 1 / 2).
    """
    ei = ELEM[w.act]
    eo = OUT_ELEM[w.act]
    flop = 0
    byt = 0
    fwd_b = 0
    bwd_b = 0
    for L in w.layers:
        r = L.ranks[L.d]
        if w.diag == "pruned_half":
            r = r - r // 2
        flop += 6 * T * r * (L.N + L.M)
    if w.ffn:
        up, dn = w.layers
        N, M = up.N, dn.M
    else:
        N, M = w.layers[0].N, w.layers[0].M
    byt = T * (2 * N * ei + M * ei + M * eo + N * eo)
    fwd_b = T * (N * ei + M * eo)
    bwd_b = T * (N * ei + M * ei + N * eo)
    return {"flop": int(flop), "bytes": int(byt), "fwd_bytes": int(fwd_b),
            "bwd_bytes": int(bwd_b)}


def all_reduce_scalar(v, op, device=None):
    """Reduce one number over all ranks ("max", "min" or "sum"); identity
    without an initialised process group.  NCCL groups reduce on the GPU,
    others (gloo) on the CPU."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return v
    dev = device if (device is not None and dist.get_backend() == "nccl") else "cpu"
    t = torch.tensor([float(v)], dtype=torch.float64, device=dev)
    ops = {"max": dist.ReduceOp.MAX, "min": dist.ReduceOp.MIN, "sum": dist.ReduceOp.SUM}
    dist.all_reduce(t, op=ops[op])
    return float(t.item())


def whole_job_rate(tokens_per_rank, world, step_ms_max):
    """Tokens of all ranks per second, timed by the slowest rank."""
    return world * tokens_per_rank / (step_ms_max * 1e-3)


SM_MAX_MHZ = 2070   # GB300 maximum SM clock


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def oracle_threads():
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 0) for i in threadpool_info()), default=0)
        if n:
            return int(n)
    except Exception:
        pass
    return os.cpu_count() or 1


def oracle_step(w, inp):
    """One fwd+bwd of the oracle over the given inputs."""
    from oracle import tt_oracle as O
    import numpy as np
    if w.ffn:
        up = ([c.astype(np.float64) for c in inp.layers[0].cores],
              [e.astype(np.float64) for e in inp.layers[0].diags])
        dn = ([c.astype(np.float64) for c in inp.layers[1].cores],
              [e.astype(np.float64) for e in inp.layers[1].diags])
        O.ffn_forward(up, dn, w.layers[0].d, w.layers[1].d, inp.x)
        O.ffn_backward(up, dn, w.layers[0].d, w.layers[1].d, inp.x, inp.dy)
    else:
        L = w.layers[0]
        cores = [c.astype(np.float64) for c in inp.layers[0].cores]
        diags = [e.astype(np.float64) for e in inp.layers[0].diags]
        O.chained_forward(cores, diags, L.d, inp.x)
        O.chained_backward(cores, diags, L.d, inp.x, inp.dy)


def time_oracle(w, sample_tokens, budget_s):
    """Run the oracle on samples of sample_tokens until budget_s has passed."""
    from tensor_train_compressed_tt_gb300 import synth
    inp = synth.draw(w, seed=0, tokens=sample_tokens)
    oracle_step(w, inp)  # warm (BLAS thread pool, page-in)
    n = 0
    t0 = time.perf_counter()
    while True:
        oracle_step(w, inp)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return n * sample_tokens / el, n, el


# ---------------------------------------------------------------------------
# clocks during the timed region


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        self.samples = []   # (host time, SM MHz)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            self.samples.append((t, sm[-1]))
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm_sorted = sorted(sm)
        return {"sm_mhz": sm_sorted[len(sm_sorted) // 2], "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm), "interval_ms": 100}

    def binned(self, windows, ms_per_step, nbins=8):
        """The timed repeats split into nbins consecutive groups: per group its
        median ms a step and the median SM clock sampled inside it."""
        out = []
        R = len(windows)
        if R == 0:
            return out
        for b in range(nbins):
            lo, hi = b * R // nbins, (b + 1) * R // nbins
            if hi <= lo:
                continue
            t0, t1 = windows[lo][0], windows[hi - 1][1]
            mhz = sorted(v for t, v in getattr(self, "samples", []) if t0 <= t <= t1)
            ms = sorted(ms_per_step[lo:hi])
            out.append({"repeats": [lo, hi], "ms_per_step": ms[len(ms) // 2],
                        "sm_mhz": mhz[len(mhz) // 2] if mhz else None, "clock_samples": len(mhz)})
        return out


def timed_repeats(run, K, barrier, stream, min_seconds, min_repeats=50, max_repeats=20000):
    """Time R repeats of the K-step region, each bracketed by a barrier and a
    device synchronise on both sides and timed by CUDA events on the launching
    stream; R >= min_repeats and the repeats together last >= min_seconds.
    Returns the per-repeat ms a step and the host time window of each repeat."""
    import torch
    evs, windows = [], []
    t_start = time.perf_counter()
    r = 0
    while r < max_repeats:
        barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        h0 = time.perf_counter()
        a.record(stream)
        for i in range(K):
            run(i)
        b.record(stream)
        barrier()
        windows.append((h0, time.perf_counter()))
        evs.append((a, b))
        r += 1
        if r >= min_repeats and time.perf_counter() - t_start >= min_seconds:
            break
    return [a.elapsed_time(b) / K for a, b in evs], windows


def spread(ms):
    """Median and spread of per-repeat times (ms a step)."""
    v = sorted(ms)
    n = len(v)
    q = lambda f: v[min(n - 1, int(f * (n - 1) + 0.5))]
    return {"repeats": n, "median": q(0.5), "min": v[0], "p10": q(0.1), "p90": q(0.9),
            "max": v[-1]}


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.split(":")[0].strip() in ("Model name", "Model"):
                v = ln.split(":", 1)[1].strip()
                if v and not v.isdigit():
                    return v
        vendor = [ln.split(":", 1)[1].strip() for ln in out.splitlines()
                  if ln.startswith("Vendor ID")]
        if vendor:
            return vendor[0]
    except Exception:
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def single_thread_rate(workload, sample, budget_s):
    """The oracle's rate on one host core: a fresh interpreter (exec, not a
    fork of this process) with every BLAS thread pool set to one thread.
    Returns (tokens/s, passes, seconds) or None."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
              "BLIS_NUM_THREADS", "VECLIB_MAXIMUM_THREADS", "NUMEXPR_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-rate",
                            "--workload", workload, "--tokens", str(sample),
                            "--target-seconds", str(budget_s)],
                           env=env, capture_output=True, text=True, timeout=10 * budget_s + 120)
        d = json.loads(r.stdout.strip().splitlines()[-1])
        return d["rate"], d["passes"], d["seconds"]
    except Exception:
        return None


def oracle_rate_main(args):
    """--oracle-rate: print the oracle's rate on this process's threads."""
    from tensor_train_compressed_tt_gb300 import synth
    if args.workload in synth.TTM_WORKLOADS:
        rate, n, el = time_ttm_oracle(synth.TTM_WORKLOADS[args.workload], args.tokens,
                                      args.target_seconds)
    else:
        rate, n, el = time_oracle(synth.WORKLOADS[args.workload], args.tokens, args.target_seconds)
    print(json.dumps({"rate": rate, "passes": n, "seconds": el}), flush=True)


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle


def graph_steps(nsets, passes, most=64):
    """Steps one graph replay runs: `passes` passes over the `nsets` rotating
    input sets, one step per set.  Each replay boundary costs a few
    microseconds (no programmatic launch edge crosses it), so a few sets get
    several passes; many small sets already amortise it, and there the graph
    keeps one pass, so that it stays short to capture."""
    return nsets * max(1, min(passes, most // nsets))


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    T_full = args.tokens or w.tokens
    K = args.steps if args.steps is not None else 20
    W = args.warmup
    # calibrate: tokens/s of the oracle on a small sample
    rate, _, _ = time_oracle(w, min(T_full, 256), 1.0)
    budget = 120.0
    per_step = budget / max(1, K + W)
    sample = int(max(16, min(T_full, rate * per_step)))
    from tensor_train_compressed_tt_gb300 import synth
    inp = synth.draw(w, seed=0, tokens=sample)
    for _ in range(W):
        oracle_step(w, inp)
    t0 = time.perf_counter()
    for _ in range(K):
        oracle_step(w, inp)
    el = time.perf_counter() - t0
    value = K * sample / el
    cores = oracle_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": K, "warmup": W, "ms_per_step": 1e3 * el / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "description": w.description, "tokens": T_full,
                   "sample_tokens_per_step": sample},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{sample} of {T_full} tokens per step, fp64 numpy oracle "
                                   f"(merged contraction order), {K} steps"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm


def gelu_rates(nsm, dev, stream):
    """Evaluations a second of the fused FFN kernels' GELU (index 0) and
    GELU + GELU' (index 1) arithmetic, from tt_gelu_rate timed with CUDA
    events: a microbenchmark of the elementwise term on every SM."""
    import torch
    from tensor_train_compressed_tt_gb300 import ttc
    blocks, iters = 8 * nsm, 2000
    out = torch.empty(blocks * 256, device=dev)
    sh = int(stream.cuda_stream)
    rates = []
    for mode in (0, 1):
        ttc.check(ttc.lib().tt_gelu_rate(mode, iters, blocks, out.data_ptr(), sh), "tt_gelu_rate")
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(3):
            ttc.check(ttc.lib().tt_gelu_rate(mode, iters, blocks, out.data_ptr(), sh),
                      "tt_gelu_rate")
        b.record(stream)
        b.synchronize()
        rates.append(3 * blocks * 256 * 16 * iters / (a.elapsed_time(b) * 1e-3))
    return rates


def traffic_for(phase_name, workload):
    """DRAM bytes per launch from the committed ncu summary, if still current."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        with open(p) as f:
            entries = json.load(f)
    except Exception:
        return None
    for e in entries:
        if e.get("phase") != phase_name or e.get("workload") != workload:
            continue
        src = os.path.join(ROOT, e["source"])
        if not os.path.exists(src):
            return None
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if sha != e.get("source_sha"):
            return None
        return e.get("dram_bytes_per_launch")
    return None


def run_ours(args, w):
    import numpy as np
    import torch

    from tensor_train_compressed_tt_gb300 import _build, synth, ttc
    from tensor_train_compressed_tt_gb300.layer import TTFFN, TTLinear

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if not os.path.exists(ttc.LIB_PATH):
        _build.build()
    T = args.tokens or w.tokens
    dt = {"bf16": torch.bfloat16, "f32": torch.float32, "e4m3": torch.uint8}[w.act]
    dto = torch.bfloat16 if w.act == "e4m3" else dt   # y and dx
    ei, eo = ELEM[w.act], OUT_ELEM[w.act]

    def to_act(a):   # float32 tensor -> the layer's input encoding
        if w.act == "e4m3":
            return a.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
        return a.to(dt)

    # ---- setup: parameters and rotating activation sets larger than 2x L2
    inp0 = synth.draw(w, seed=rank, tokens=T)
    if w.ffn:
        up, dn = w.layers
        mod = TTFFN((up.in_modes, up.out_modes, up.ranks), (dn.in_modes, dn.out_modes, dn.ranks),
                    dt, reuse_merge=not args.no_reuse,
                    reuse_z=not (args.no_reuse or args.no_reuse_z),
                    deterministic=args.deterministic)
        params = [torch.from_numpy(synth.pack(l.cores, l.diags)).to(dev) for l in inp0.layers]
        N, M = up.N, dn.M
        n_par = [p.numel() for p in params]
    else:
        L = w.layers[0]
        mod = TTLinear(L.in_modes, L.out_modes, L.ranks, dt, reuse_merge=not args.no_reuse,
                       reuse_z=not (args.no_reuse or args.no_reuse_z),
                       deterministic=args.deterministic)
        params = [torch.from_numpy(synth.pack(inp0.layers[0].cores, inp0.layers[0].diags)).to(dev)]
        N, M = L.N, L.M
        n_par = [params[0].numel()]
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    set_bytes = T * (N + M) * (ei + eo)
    nsets = max(2, -(-2 * l2 // set_bytes) + 1)
    sets = []
    for i in range(nsets):
        g = torch.Generator(device=dev)
        g.manual_seed(1000 * rank + i)
        x = to_act(torch.randn((T, N), generator=g, device=dev, dtype=torch.float32))
        dy = to_act(torch.randn((T, M), generator=g, device=dev, dtype=torch.float32))
        y = torch.empty((T, M), device=dev, dtype=dto)
        dx = torch.empty((T, N), device=dev, dtype=dto)
        sets.append((x, dy, y, dx))
    # the first set holds the seeded synthetic inputs of the workload
    if w.act == "e4m3":
        sets[0][0].copy_(torch.from_numpy(synth.e4m3_bytes(inp0.x)).to(dev))
        sets[0][1].copy_(torch.from_numpy(synth.e4m3_bytes(inp0.dy)).to(dev))
    else:
        sets[0][0].copy_(torch.from_numpy(inp0.x).to(dev).to(dt))
        sets[0][1].copy_(torch.from_numpy(inp0.dy).to(dev).to(dt))
    dparams = [torch.empty(n, device=dev, dtype=torch.float32) for n in n_par]
    ws = mod.workspace(T, dev)
    stream = torch.cuda.current_stream(dev)
    sh = int(stream.cuda_stream)
    wsp, wsn = ws.data_ptr(), ws.numel()

    def run_step(x, dy, y, dx, dps, sh):
        """One fwd+bwd step through the C ABI on the given device buffers."""
        if w.ffn:
            ttc.check(ttc.tt_ffn_forward(mod.plan, T, x.data_ptr(), params[0].data_ptr(),
                                         params[1].data_ptr(), y.data_ptr(), wsp, wsn, sh))
            ttc.check(ttc.tt_ffn_backward(mod.plan, T, x.data_ptr(), dy.data_ptr(),
                                          params[0].data_ptr(), params[1].data_ptr(),
                                          dx.data_ptr(), dps[0].data_ptr(),
                                          dps[1].data_ptr(), wsp, wsn, sh))
        else:
            ttc.check(ttc.tt_forward(mod.plan, T, x.data_ptr(), params[0].data_ptr(),
                                     y.data_ptr(), wsp, wsn, sh))
            ttc.check(ttc.tt_backward(mod.plan, T, x.data_ptr(), dy.data_ptr(),
                                      params[0].data_ptr(), dx.data_ptr(),
                                      dps[0].data_ptr(), wsp, wsn, sh))

    def step(i, sh=sh):
        x, dy, y, dx = sets[i % nsets]
        run_step(x, dy, y, dx, dparams, sh)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    W = max(3, args.warmup)
    for i in range(W):
        step(i)
    ttc.check(ttc.tt_get_device_status(sh), "device status after warm-up")
    barrier()

    # One CUDA graph holds one pass over the rotating input sets: nsets whole
    # fwd+bwd steps in a row, as the CoMERA pages capture their training step
    # in a graph.  Inside a graph consecutive steps keep the programmatic
    # (PDL) edges between their kernels; --eager launches from the host every
    # time instead.
    graph, graph_note, launches_per_step = None, "eager", None
    gsteps = graph_steps(nsets, args.graph_passes)
    if not args.eager:
        try:
            g = torch.cuda.CUDAGraph()
            c0 = ttc.lib().tt_launch_count()
            with torch.cuda.graph(g):
                cs = int(torch.cuda.current_stream().cuda_stream)
                for j in range(gsteps):
                    step(j, cs)
            launches_per_step = int(ttc.lib().tt_launch_count() - c0) // gsteps
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize(dev)
            ttc.check(ttc.tt_get_device_status(sh), "device status after graph warm-up")
            graph = g
            graph_note = (f"cuda_graph ({gsteps} steps per replay: {gsteps // nsets} "
                          f"pass{'es' if gsteps > nsets else ''} over "
                          f"the {nsets} rotating input sets)")
        except Exception as e:  # capture unsupported: time the eager loop
            graph, graph_note = None, f"eager (graph capture failed: {type(e).__name__}: {e})"
            torch.cuda.synchronize(dev)

    def run(i):
        """Step i; with the graph, a replay runs steps i .. i + gsteps - 1."""
        if graph is not None:
            if i % gsteps == 0:
                graph.replay()
        else:
            step(i)
    # K steps a timed region (whole graph replays); the region is repeated
    # until the repeats last target-seconds (at least 50 of them), and the
    # median repeat gives ms_per_step
    K = args.steps if args.steps is not None else 20
    if graph is not None:
        K = -(-K // gsteps) * gsteps   # whole replays
    barrier()

    # ---- timed region
    uuid = getattr(props, "uuid", None)
    clocks = ClockSampler(f"GPU-{uuid}" if uuid is not None else str(local))
    clocks.start()
    time.sleep(0.3)
    l0 = ttc.lib().tt_launch_count()
    rep_ms, windows = timed_repeats(run, K, barrier, stream, args.target_seconds)
    launches = int(ttc.lib().tt_launch_count() - l0) // len(rep_ms)
    if graph is not None:
        launches = K * launches_per_step  # replays launch without the host counter
    clk = clocks.stop()
    if clk is not None:
        clk["by_repeat_group"] = clocks.binned(windows, rep_ms)
    rep = spread(rep_ms)
    ms = all_reduce_scalar(rep["median"], "max", dev)
    ttc.check(ttc.tt_get_device_status(sh), "device status after timed region")

    # the same steps launched eagerly, for reference
    Ke = min(K, 2000)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(Ke):
        step(i)
    e1.record(stream)
    barrier()
    ms_eager = all_reduce_scalar(e0.elapsed_time(e1) / Ke, "max", dev)

    # ---- per-phase CUDA-event timing of the library's kernels (same steps):
    # the library brackets each kernel phase with events on the launching
    # stream.  Eagerly launched, the events also take in the host's launch
    # latency; inside a replayed graph (event-record nodes) they time each
    # kernel from the end of the node before it, as the timed region runs them.
    import ctypes

    def read_phases(acc):
        for ph in range(5):
            tot = ctypes.c_double()
            n = ctypes.c_int64()
            ttc.check(ttc.lib().tt_profile_phase(ph, ctypes.byref(tot), ctypes.byref(n)))
            name = ttc.lib().tt_profile_phase_name(ph)
            name = name.decode() if isinstance(name, bytes) else str(name)
            if n.value:
                a = acc.setdefault(name, {"ms_total": 0.0, "intervals": 0})
                a["ms_total"] += tot.value
                a["intervals"] += n.value
        for a in acc.values():
            a["us_per_interval"] = 1e3 * a["ms_total"] / a["intervals"]
        return acc

    ttc.lib().tt_profile_enable(1)
    barrier()
    for i in range(K):
        step(i)
    barrier()
    phases_eager = read_phases({})
    ttc.lib().tt_profile_enable(0)
    phases, phase_note = phases_eager, "eager launches with events between them"
    if graph is not None:
        try:
            ttc.lib().tt_profile_enable(1)
            gp = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gp):
                cs = int(torch.cuda.current_stream().cuda_stream)
                for j in range(nsets):
                    step(j, cs)
            ttc.lib().tt_profile_enable(0)
            gp.replay()
            torch.cuda.synchronize(dev)
            acc = {}
            for _ in range(max(10, K // nsets)):
                gp.replay()
                torch.cuda.synchronize(dev)
                read_phases(acc)
            phases, phase_note = acc, "graph replays with event-record nodes around each phase"
        except Exception as e:  # keep the eager figures
            ttc.lib().tt_profile_enable(0)
            phase_note = f"eager ({type(e).__name__} in the graph pass: {e})"
            torch.cuda.synchronize(dev)

    # ---- the rank-adaptive step (proximal update of one layer's packed
    # parameters), timed on copies so the step's own buffers stay unchanged
    rank_step = None
    if not w.ffn:
        pc = params[0].clone()
        gc = dparams[0].clone()
        n_up = 200
        for _ in range(3):
            ttc.check(ttc.tt_rank_update(mod.plan, pc.data_ptr(), gc.data_ptr(), 1e-3, 1e-3,
                                         1e-3, sh), "tt_rank_update")
        barrier()
        r0 = torch.cuda.Event(enable_timing=True)
        r1 = torch.cuda.Event(enable_timing=True)
        r0.record(stream)
        for _ in range(n_up):
            ttc.check(ttc.tt_rank_update(mod.plan, pc.data_ptr(), gc.data_ptr(), 1e-3, 1e-3,
                                         1e-3, sh), "tt_rank_update")
        r1.record(stream)
        barrier()
        us = 1e3 * r0.elapsed_time(r1) / n_up
        nb = 12 * pc.numel()  # read params and dparams, write params (float32)
        # the same step fused into the backward's merge program: the added
        # time of tt_backward_rank_update over tt_backward (gradient form, so
        # the parameters stay as they are)
        x0, dy0, _, dx0 = sets[0]

        def bwd_time(fused, n=50):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            barrier()
            a.record(stream)
            for _ in range(n):
                if fused:
                    ttc.check(ttc.tt_backward_rank_update(
                        mod.plan, T, x0.data_ptr(), dy0.data_ptr(), pc.data_ptr(), dx0.data_ptr(),
                        gc.data_ptr(), 1e-3, 1e-3, 0.0, wsp, wsn, sh))
                else:
                    ttc.check(ttc.tt_backward(mod.plan, T, x0.data_ptr(), dy0.data_ptr(),
                                              pc.data_ptr(), dx0.data_ptr(), gc.data_ptr(), wsp,
                                              wsn, sh))
            b.record(stream)
            barrier()
            return 1e3 * a.elapsed_time(b) / n
        ttc.check(ttc.tt_forward(mod.plan, T, x0.data_ptr(), pc.data_ptr(), sets[0][2].data_ptr(),
                                 wsp, wsn, sh))
        t_b, t_bf = bwd_time(False), bwd_time(True)
        rank_step = {"us_per_call": us, "bytes_per_call": nb,
                     "achieved_gbs": nb / (us * 1e-6) / 1e9, "bound": "latency",
                     "note": "tt_rank_update, proximal step on one layer's packed "
                             f"parameters ({pc.numel()} floats), back-to-back eager launches",
                     "fused_added_us": t_bf - t_b, "backward_us": t_b,
                     "backward_with_step_us": t_bf,
                     "fused_note": "tt_backward_rank_update (the step as the last phase of the "
                                   "merge program) against tt_backward, eager, 50 calls each"}

    alg = algorithmic(w, T)
    peak, peak_kind = measured_peaks()
    # A step whose HBM time is under a microsecond is bound by kernel
    # launches: its floor is the same step on one token, replayed the same way
    launch_floor = None
    if alg["bytes"] / (peak * 1e9) < 1e-6:
        x1, dy1 = sets[0][0][:1].contiguous(), sets[0][1][:1].contiguous()
        y1, dx1 = sets[0][2][:1].contiguous(), sets[0][3][:1].contiguous()

        def step1(i, sh=sh):
            x, dy, y, dx = x1, dy1, y1, dx1
            ttc.check(ttc.tt_forward(mod.plan, 1, x.data_ptr(), params[0].data_ptr(),
                                     y.data_ptr(), wsp, wsn, sh))
            ttc.check(ttc.tt_backward(mod.plan, 1, x.data_ptr(), dy.data_ptr(),
                                      params[0].data_ptr(), dx.data_ptr(),
                                      dparams[0].data_ptr(), wsp, wsn, sh))
        run1 = step1
        if graph is not None:
            g1 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g1):
                cs = int(torch.cuda.current_stream().cuda_stream)
                for j in range(gsteps):
                    step1(j, cs)
            for _ in range(3):
                g1.replay()

            def run1(i):
                if i % gsteps == 0:
                    g1.replay()
        ms1 = spread(timed_repeats(run1, K, barrier, stream, 0.3)[0])["median"]
        launch_floor = {"ms_per_step_1_token": ms1, "launches_per_step": launches_per_step,
                        "note": "the same step on 1 token, replayed the same way: the launch "
                                "floor of this path"}
    bytes_of = {"forward_tokens": alg["fwd_bytes"], "backward_tokens": alg["bwd_bytes"]}
    dom = None
    for nm in ("backward_tokens", "forward_tokens"):
        if nm in phases and (dom is None or phases[nm]["ms_total"] > phases[dom]["ms_total"]):
            dom = nm
    roof = None
    if dom is not None:
        per_launch_s = phases[dom]["us_per_interval"] * 1e-6
        fused_ffn = w.ffn and not args.deterministic
        if w.ffn and not fused_ffn:
            per_launch_s *= 2  # two layers bracketed per pass; bytes cover the pair
        if fused_ffn:
            # The fused pair's floor is not HBM: every hidden activation takes
            # one tanh on the special-function units (GELU in the forward, GELU
            # and GELU' in the backward), T x H evaluations a launch, against
            # 16 a clock per SM at the maximum SM clock.
            H = w.layers[0].M
            evals = T * H
            sfu_peak = 16 * props.multi_processor_count * SM_MAX_MHZ * 1e6
            ach = evals / per_launch_s
            roof = {"bound": "alu", "kernel": dom, "achieved": ach / 1e9, "peak": sfu_peak / 1e9,
                    "peak_kind": "derived: 16 special-function results a clock per SM x "
                                 f"{props.multi_processor_count} SMs x {SM_MAX_MHZ} MHz",
                    "unit": "G tanh/s", "frac": ach / sfu_peak, "traffic": None,
                    "algorithmic_evals_per_launch": evals, "duration_us": per_launch_s * 1e6,
                    "hbm_frac": bytes_of[dom] / per_launch_s / 1e9 / peak,
                    "timing": phase_note}
            # the GELU term measured: the kernels' own packed GELU (forward)
            # and GELU + GELU' (backward) arithmetic, in registers on every SM
            rates = gelu_rates(props.multi_processor_count, dev, stream)
            gm = {"unit": "G evaluations/s", "note": "tt_gelu_rate: 8 blocks of 256 threads an "
                  "SM, 16 values a thread, 2000 rounds, CUDA events; floor = T x 3072 / rate"}
            for nm, mode in (("forward_tokens", 0), ("backward_tokens", 1)):
                floor_s = evals / rates[mode]
                gm[nm] = {"rate": rates[mode] / 1e9, "floor_us": floor_s * 1e6}
                if nm in phases:
                    gm[nm]["frac"] = floor_s / (phases[nm]["us_per_interval"] * 1e-6)
            roof["gelu_measured"] = gm
        else:
            ach = bytes_of[dom] / per_launch_s / 1e9
            roof = {"bound": "hbm", "kernel": dom, "achieved": ach, "peak": peak,
                    "peak_kind": peak_kind, "unit": "GB/s", "frac": ach / peak,
                    "traffic": traffic_for(dom, w.name),
                    "algorithmic_bytes_per_launch": bytes_of[dom],
                    "duration_us": per_launch_s * 1e6, "timing": phase_note}
    if launch_floor is not None:
        # launch-bound: the achieved step rate against the 1-token step rate
        roof = {"bound": "launch", "kernel": "whole step", "achieved": 1e3 / ms,
                "peak": 1e3 / launch_floor["ms_per_step_1_token"], "unit": "steps/s",
                "frac": launch_floor["ms_per_step_1_token"] / ms, "traffic": None,
                "note": "HBM time of the step is nanoseconds; the bound is the launch floor "
                        "(the same step on 1 token)"}
    t_roof = alg["bytes"] / (peak * 1e9)
    value = whole_job_rate(T, world, ms)

    # ---- end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        # Every step copies its inputs (x, dy) in from pinned host memory and
        # reads its result back: the parameter gradients (dparams), which is
        # what a training step hands on; y and dx feed the neighbouring layers
        # on the device.  The copies run on their own streams into two
        # alternating device buffer sets, so step i+1's host->device copy and
        # step i-1's device->host copy overlap step i's kernels.  The same
        # pipeline that also reads y and dx back to the host is measured too
        # (with_activations_out).
        x0, dy0, y0, dx0 = sets[0]
        hx = torch.empty(x0.shape, dtype=dt, pin_memory=True)
        hdy = torch.empty(dy0.shape, dtype=dt, pin_memory=True)
        hy = torch.empty(y0.shape, dtype=dto, pin_memory=True)
        hdx = torch.empty(dx0.shape, dtype=dto, pin_memory=True)
        hdp = [torch.empty(n, dtype=torch.float32, pin_memory=True) for n in n_par]
        hx.copy_(x0)
        hdy.copy_(dy0)
        dparams2 = [torch.empty(n, device=dev, dtype=torch.float32) for n in n_par]
        bufs = [sets[0] + (dparams,), sets[1] + (dparams2,)]
        s_in = torch.cuda.Stream(dev)
        s_out = torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        Ke = max(3, min(K, 200))

        def e2e_step(i, acts_out):
            j = i % 2
            x, dy, y, dx, dps = bufs[j]
            s_in.wait_event(ev_done[j])          # the step that last read set j is done
            with torch.cuda.stream(s_in):
                x.copy_(hx, non_blocking=True)
                dy.copy_(hdy, non_blocking=True)
            ev_in[j].record(s_in)
            stream.wait_event(ev_in[j])
            stream.wait_event(ev_out[j])         # set j's last results are read out
            run_step(x, dy, y, dx, dps, sh)
            ev_done[j].record(stream)
            s_out.wait_event(ev_done[j])
            with torch.cuda.stream(s_out):
                if acts_out:
                    hy.copy_(y, non_blocking=True)
                    hdx.copy_(dx, non_blocking=True)
                for hp, dp in zip(hdp, dps):
                    hp.copy_(dp, non_blocking=True)
            ev_out[j].record(s_out)

        def e2e_ms(acts_out):
            for i in range(3):
                e2e_step(i, acts_out)
            torch.cuda.synchronize(dev)
            barrier()
            a0 = torch.cuda.Event(enable_timing=True)
            a1 = torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            s_in.wait_event(a0)
            for i in range(Ke):
                e2e_step(i, acts_out)
            stream.wait_event(ev_out[(Ke - 1) % 2])  # the last step's results are on the host
            a1.record(stream)
            barrier()
            return all_reduce_scalar(a0.elapsed_time(a1) / Ke, "max", dev)

        h2d = int(hx.numel() * ei + hdy.numel() * ei)
        d2h_p = int(4 * sum(n_par))
        d2h_a = int(hy.numel() * eo + hdx.numel() * eo)
        ems = e2e_ms(False)
        ems_a = e2e_ms(True)
        e2e = {"value": whole_job_rate(T, world, ems), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h_p,
               "ms_per_step": ems, "steps": Ke,
               "pipeline": "x, dy in and dparams out every step, on copy streams of their "
                           "own, two device buffer sets",
               "with_activations_out": {"value": whole_job_rate(T, world, ems_a),
                                        "d2h_bytes_per_step": d2h_p + d2h_a,
                                        "ms_per_step": ems_a,
                                        "note": "the same pipeline also reading y and dx back"}}

    # ---- oracle on the host cores (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sample = min(T, 2048)
        rate, n, el = time_oracle(w, sample, 10.0)
        one = single_thread_rate(w.name, min(T, 512), 8.0)
        cpu = {"value": rate, "unit": "tokens/s", "cores": oracle_threads(), "kind": "oracle",
               "cpu_model": cpu_model(), "nproc": os.cpu_count(),
               "sample": f"{n} fwd+bwd passes of the fp64 numpy oracle on {sample} of the "
                         f"{T} tokens ({el:.1f} s)",
               "single_thread": None if one is None else
               {"value": one[0], "unit": "tokens/s", "cores": 1,
                "sample": f"{one[1]} passes on {min(T, 512)} tokens ({one[2]:.1f} s)"}}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.act, "data": "synthetic",
            "timing": dict(rep, note="ms_per_step is the median over repeats of the K-step "
                                     "region, max over ranks"),
            "config": {"workload": w.name, "description": w.description, "tokens": T,
                       "modes": [list(L.modes) for L in w.layers],
                       "ranks": [list(L.ranks) for L in w.layers],
                       "l2": f"{nsets} rotating input/output sets of {set_bytes / 1e6:.1f} MB "
                             f"(> 2x L2 of {l2 / 1e6:.0f} MB)",
                       "parallelism": f"replicas x{world}",
                       "reuse_merge": not args.no_reuse,
                       "reuse_z": not (args.no_reuse or args.no_reuse_z) and w.act != "f32",
                       "deterministic": bool(args.deterministic),
                       "launch": graph_note},
            "ms_per_step_eager": ms_eager,
            "roofline": roof,
            "roofline_step": {"t_roof_us": t_roof * 1e6, "frac": t_roof / (ms * 1e-3),
                              "algorithmic_bytes": alg["bytes"], "algorithmic_flop": alg["flop"],
                              "peak_gbs": peak, "peak_kind": peak_kind},
            "phases_us": {k: round(v["us_per_interval"], 3) for k, v in phases.items()},
            "phases_us_eager": {k: round(v["us_per_interval"], 3) for k, v in phases_eager.items()},
            "phases_timing": phase_note,
            "rank_update": rank_step,
            "launch_floor": launch_floor,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# TT-matrix embedding lookup (a second workload: lookup + backward per step)


def ttm_oracle_step(inp):
    from oracle import tt_oracle as O
    import numpy as np
    cores = [c.astype(np.float64) for c in inp.cores]
    diags = [e.astype(np.float64) for e in inp.diags]
    O.ttm_lookup(cores, diags, inp.idx)
    O.ttm_lookup_backward(cores, diags, inp.idx, inp.dout)


def time_ttm_oracle(w, sample, budget_s):
    from tensor_train_compressed_tt_gb300 import synth
    inp = synth.draw_ttm(w, seed=0, batch=sample)
    ttm_oracle_step(inp)
    n = 0
    t0 = time.perf_counter()
    while True:
        ttm_oracle_step(inp)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return n * sample / el, n, el


def run_ttm(args, w):
    """Lookup + backward of a TT-matrix table per step (graph-replayed)."""
    import numpy as np
    import torch

    from tensor_train_compressed_tt_gb300 import _build, synth, ttc
    from tensor_train_compressed_tt_gb300.layer import TTMEmbedding

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if not os.path.exists(ttc.LIB_PATH):
        _build.build()
    B = args.tokens or w.batch
    S = w.shape
    inp0 = synth.draw_ttm(w, seed=rank, batch=B)
    # the step's backward takes the distinct rows its lookup found (TT_REUSE_MERGE)
    emb = TTMEmbedding(S.row_modes, S.col_modes, S.ranks, reuse=True)
    params = torch.from_numpy(synth.pack(inp0.cores, inp0.diags)).to(dev)
    dparams = torch.empty(emb.n_params, device=dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    set_bytes = 4 * B * (2 * S.Dm + 1)
    nsets = max(2, -(-2 * l2 // set_bytes) + 1)
    sets = []
    for i in range(nsets):
        t = inp0 if i == 0 else synth.draw_ttm(w, seed=1000 * rank + i, batch=B)
        sets.append((torch.from_numpy(t.idx).to(dev), torch.from_numpy(t.dout).to(dev),
                     torch.empty((B, S.Dm), device=dev)))
    ws = emb.workspace(B, dev)
    stream = torch.cuda.current_stream(dev)
    sh = int(stream.cuda_stream)
    wsp, wsn = ws.data_ptr(), ws.numel()

    def fwd(i, sh=sh):
        idx, _, out = sets[i % nsets]
        ttc.check(ttc.tt_ttm_lookup(emb.plan, B, idx.data_ptr(), params.data_ptr(),
                                    out.data_ptr(), wsp, wsn, sh))

    def bwd(i, sh=sh):
        idx, dout, _ = sets[i % nsets]
        ttc.check(ttc.tt_ttm_lookup_backward(emb.plan, B, idx.data_ptr(), dout.data_ptr(),
                                             params.data_ptr(), dparams.data_ptr(), wsp, wsn,
                                             sh))

    def step(i, sh=sh):
        fwd(i, sh)
        bwd(i, sh)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    W = max(3, args.warmup)
    for i in range(W):
        step(i)
    ttc.check(ttc.tt_get_device_status(sh), "device status after warm-up")
    barrier()
    uniq, pairs = emb.stats(ws)
    graph, graph_note, per_step = None, "eager", None
    gsteps = graph_steps(nsets, args.graph_passes)
    if not args.eager:
        try:
            g = torch.cuda.CUDAGraph()
            c0 = ttc.lib().tt_launch_count()
            with torch.cuda.graph(g):
                cs = int(torch.cuda.current_stream().cuda_stream)
                for j in range(gsteps):
                    step(j, cs)
            per_step = int(ttc.lib().tt_launch_count() - c0) // gsteps
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize(dev)
            graph, graph_note = g, (f"cuda_graph ({gsteps} steps per replay: {gsteps // nsets} "
                                    f"pass{'es' if gsteps > nsets else ''} over the {nsets} input sets)")
        except Exception as e:
            graph, graph_note = None, f"eager (graph capture failed: {type(e).__name__}: {e})"
            torch.cuda.synchronize(dev)

    def run(i):
        if graph is not None:
            if i % gsteps == 0:
                graph.replay()
        else:
            step(i)
    K = args.steps if args.steps is not None else 20
    if graph is not None:
        K = -(-K // gsteps) * gsteps
    barrier()
    uuid = getattr(props, "uuid", None)
    clocks = ClockSampler(f"GPU-{uuid}" if uuid is not None else str(local))
    clocks.start()
    time.sleep(0.3)
    l0 = ttc.lib().tt_launch_count()
    rep_ms, windows = timed_repeats(run, K, barrier, stream, args.target_seconds)
    launches = int(ttc.lib().tt_launch_count() - l0) // len(rep_ms)
    if graph is not None:
        launches = K * per_step
    clk = clocks.stop()
    if clk is not None:
        clk["by_repeat_group"] = clocks.binned(windows, rep_ms)
    rep = spread(rep_ms)
    ms = all_reduce_scalar(rep["median"], "max", dev)
    ttc.check(ttc.tt_get_device_status(sh), "device status after timed region")

    # each call on its own (eager), for the roofline of the dominant one
    def timed(fn, n=50):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        barrier()
        a.record(stream)
        for i in range(n):
            fn(i)
        b.record(stream)
        barrier()
        return a.elapsed_time(b) / n * 1e-3
    # (the backward of a plan that reuses the lookup's bookkeeping follows the
    # lookup of its own batch: its time is a lookup + backward pair's less
    # the lookup's)
    t_f = timed(fwd)
    t_b = timed(step) - t_f
    peak, peak_kind = measured_peaks()
    # algorithmic bytes: lookup writes B x Dm rows and reads the indices;
    # backward reads dout and the indices (tables and gradients: < 1 MB)
    by_f = 4 * B * (S.Dm + 1)
    by_b = 4 * B * (S.Dm + 1)
    dom, t_dom, by_dom = ("backward", t_b, by_b) if t_b >= t_f else ("lookup", t_f, by_f)
    ach = by_dom / t_dom / 1e9
    roof = {"bound": "hbm", "kernel": f"tt_ttm_{dom} (one call, several kernels)",
            "achieved": ach, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
            "frac": ach / peak, "traffic": None, "algorithmic_bytes_per_launch": by_dom}
    value = whole_job_rate(B, world, ms)

    e2e = None
    if not args.no_e2e:
        # every step: the indices and dout in from pinned host memory, the
        # step's result (dparams) out; the looked-up rows feed the model on
        # the device (the same loop also reading them back: with_rows_out)
        hi = torch.from_numpy(inp0.idx).pin_memory()
        hd = torch.from_numpy(inp0.dout).pin_memory()
        ho = torch.empty((B, S.Dm)).pin_memory()
        hp = torch.empty(emb.n_params).pin_memory()
        di, dd, do = sets[0]
        Ke = 50

        def e2e_ms(rows_out):
            barrier()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(Ke):
                di.copy_(hi, non_blocking=True)
                dd.copy_(hd, non_blocking=True)
                fwd(0)
                bwd(0)
                if rows_out:
                    ho.copy_(do, non_blocking=True)
                hp.copy_(dparams, non_blocking=True)
            b.record(stream)
            barrier()
            return all_reduce_scalar(a.elapsed_time(b) / Ke, "max", dev)

        ms_e = e2e_ms(False)
        ms_r = e2e_ms(True)
        e2e = {"value": whole_job_rate(B, world, ms_e), "unit": "tokens/s",
               "h2d_bytes_per_step": hi.numel() * 4 + hd.numel() * 4,
               "d2h_bytes_per_step": hp.numel() * 4, "ms_per_step": ms_e, "steps": Ke,
               "with_rows_out": {"value": whole_job_rate(B, world, ms_r),
                                 "d2h_bytes_per_step": ho.numel() * 4 + hp.numel() * 4,
                                 "ms_per_step": ms_r}}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, n, el = time_ttm_oracle(w, min(B, 4000), 10.0)
        one = single_thread_rate(w.name, min(B, 1000), 8.0)
        cpu = {"value": rate, "unit": "tokens/s", "cores": oracle_threads(), "kind": "oracle",
               "cpu_model": cpu_model(), "nproc": os.cpu_count(),
               "sample": f"{n} lookup+backward passes of the fp64 numpy oracle on "
                         f"{min(B, 4000)} of the {B} indices ({el:.1f} s)",
               "single_thread": None if one is None else
               {"value": one[0], "unit": "tokens/s", "cores": 1,
                "sample": f"{one[1]} passes on {min(B, 1000)} indices ({one[2]:.1f} s)"}}
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "timing": dict(rep, note="ms_per_step is the median over repeats of the K-step "
                                     "region, max over ranks"),
            "config": {"workload": w.name, "description": w.description, "tokens": B,
                       "row_modes": list(S.row_modes), "col_modes": list(S.col_modes),
                       "ranks": list(S.ranks), "distinct_rows": uniq, "distinct_prefixes": pairs,
                       "l2": f"{nsets} rotating index/gradient/output sets of "
                             f"{set_bytes / 1e6:.1f} MB (> 2x L2 of {l2 / 1e6:.0f} MB)",
                       "parallelism": f"replicas x{world}", "launch": graph_note},
            "lookup_us": t_f * 1e6, "backward_us": t_b * 1e6,
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_ttm_reference(args, w):
    _, rank, _ = dist_env()
    if rank != 0:
        return
    B = args.tokens or w.batch
    K = args.steps if args.steps is not None else 20
    W = args.warmup
    rate, _, _ = time_ttm_oracle(w, min(B, 512), 1.0)
    per_step = 120.0 / max(1, K + W)
    sample = int(max(16, min(B, rate * per_step)))
    from tensor_train_compressed_tt_gb300 import synth
    inp = synth.draw_ttm(w, seed=0, batch=sample)
    for _ in range(W):
        ttm_oracle_step(inp)
    t0 = time.perf_counter()
    for _ in range(K):
        ttm_oracle_step(inp)
    el = time.perf_counter() - t0
    value = K * sample / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": K, "warmup": W, "ms_per_step": 1e3 * el / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "description": w.description, "tokens": B,
                   "sample_tokens_per_step": sample},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle_threads(),
                         "kind": "oracle",
                         "sample": f"{sample} of {B} indices per step, fp64 numpy oracle "
                                   f"(distinct rows only), {K} steps"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# The TT layers of one encoder block (Q, K, V, O and the FFN pair) as one step


def encoder_oracle_step(inp):
    from oracle import tt_oracle as O
    import numpy as np

    def f64(li):
        return ([c.astype(np.float64) for c in li.cores], [e.astype(np.float64) for e in li.diags])
    xin = {"q": inp.x, "k": inp.x, "v": inp.x, "o": inp.xo}
    for nm in ("q", "k", "v", "o"):
        c, d = f64(inp.layers[nm])
        O.chained_forward(c, d, 3, xin[nm])
        O.chained_backward(c, d, 3, xin[nm], inp.dy[nm])
    up, dn = f64(inp.layers["up"]), f64(inp.layers["down"])
    O.ffn_forward(up, dn, 3, 3, inp.xf)
    O.ffn_backward(up, dn, 3, 3, inp.xf, inp.dy["ffn"])


def run_encoder(args):
    import torch

    from tensor_train_compressed_tt_gb300 import _build, synth, ttc
    from tensor_train_compressed_tt_gb300.encoder import TTEncoderBlock

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if not os.path.exists(ttc.LIB_PATH):
        _build.build()
    T = args.tokens or 16384
    inp = synth.draw_encoder(T, seed=rank)
    blk = TTEncoderBlock(deterministic=args.deterministic, fuse_qkv=not args.no_fuse_qkv)
    params = {nm: torch.from_numpy(synth.pack(li.cores, li.diags)).to(dev)
              for nm, li in inp.layers.items()}
    b = blk.buffers(T, dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    set_bytes = T * 768 * 2 * 8 + 8 * T * 768 * 2   # 8 inputs, 8 outputs of 768 columns, bf16
    nsets = max(2, -(-2 * l2 // set_bytes) + 1)
    sets = []
    for i in range(nsets):
        if i == 0:
            d = lambda a: torch.from_numpy(a).to(dev).bfloat16()  # noqa: E731
            sets.append((d(inp.x), d(inp.xo), d(inp.xf), {k: d(v) for k, v in inp.dy.items()}))
            continue
        g = torch.Generator(device=dev)
        g.manual_seed(1000 * rank + i)
        r = lambda: torch.randn((T, 768), generator=g, device=dev).bfloat16()  # noqa: E731
        sets.append((r(), r(), r(), {k: r() for k in ("q", "k", "v", "o", "ffn")}))
    stream = torch.cuda.current_stream(dev)

    def step(i):
        x, xo, xf, dy = sets[i % nsets]
        blk.step(x, xo, xf, dy, params, b)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    W = max(3, args.warmup)
    for i in range(W):
        step(i)
    ttc.check(ttc.tt_get_device_status(int(stream.cuda_stream)), "device status after warm-up")
    barrier()
    graph, note, per_step = None, "eager", None
    gsteps = graph_steps(nsets, args.graph_passes)
    if not args.eager:
        g = torch.cuda.CUDAGraph()
        c0 = ttc.lib().tt_launch_count()
        with torch.cuda.graph(g):
            for j in range(gsteps):
                step(j)
        per_step = int(ttc.lib().tt_launch_count() - c0) // gsteps
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize(dev)
        graph, note = g, (f"cuda_graph ({gsteps} block steps per replay: {gsteps // nsets} "
                          f"pass{'es' if gsteps > nsets else ''} over the {nsets} input sets)")

    def run(i):
        if graph is not None:
            if i % gsteps == 0:
                graph.replay()
        else:
            step(i)
    K = args.steps if args.steps is not None else 8
    if graph is not None:
        K = -(-K // gsteps) * gsteps
    barrier()
    uuid = getattr(props, "uuid", None)
    clocks = ClockSampler(f"GPU-{uuid}" if uuid is not None else str(local))
    clocks.start()
    time.sleep(0.3)
    l0 = ttc.lib().tt_launch_count()
    rep_ms, windows = timed_repeats(run, K, barrier, stream, args.target_seconds)
    launches = int(ttc.lib().tt_launch_count() - l0) // len(rep_ms)
    if graph is not None:
        launches = K * per_step
    clk = clocks.stop()
    if clk is not None:
        clk["by_repeat_group"] = clocks.binned(windows, rep_ms)
    rep = spread(rep_ms)
    ms = all_reduce_scalar(rep["median"], "max", dev)
    ttc.check(ttc.tt_get_device_status(int(stream.cuda_stream)), "device status after timing")
    peak, peak_kind = measured_peaks()
    # summed algorithmic work of the block's TT layers: per input x read by
    # both passes and its dx written once (Q, K and V share theirs), per layer
    # dy read and y written (bf16), and 6 T r (N + M) FLOP a layer
    byts, flop = 0, 0
    for nm in ("q", "k", "v", "o"):
        sh = synth.ENCODER_LAYERS[nm]
        byts += 2 * T * 2 * sh.M
        if nm in ("q", "o"):
            byts += 2 * T * 3 * sh.N
        flop += 6 * T * sh.ranks[sh.d] * (sh.N + sh.M)
    byts += 2 * T * (3 * 768 + 2 * 768)   # the FFN pair: x, y, dy, dx of the pair
    for nm in ("up", "down"):
        sh = synth.ENCODER_LAYERS[nm]
        flop += 6 * T * sh.ranks[sh.d] * (sh.N + sh.M)
    t_roof = byts / (peak * 1e9)
    value = whole_job_rate(T, world, ms)
    # end to end: every step copies the block's eight inputs (x, xo, xf and the
    # five upstream gradients) in from pinned host memory and reads every
    # layer's dparams back, in stream order with the kernels
    e2e = None
    if not args.no_e2e:
        x0, xo0, xf0, dy0 = sets[0]
        dev_in = [x0, xo0, xf0] + [dy0[k] for k in sorted(dy0)]
        host_in = [t.cpu().pin_memory() for t in dev_in]
        dps = [b[k] for k in sorted(b) if k.startswith("dp_")]
        host_dp = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in dps]
        Ke = 8

        def e2e_run():
            for hi, di in zip(host_in, dev_in):
                di.copy_(hi, non_blocking=True)
            blk.step(x0, xo0, xf0, dy0, params, b)
            for hd, dd in zip(host_dp, dps):
                hd.copy_(dd, non_blocking=True)

        e2e_run()
        barrier()
        ea = torch.cuda.Event(enable_timing=True)
        eb = torch.cuda.Event(enable_timing=True)
        ea.record(stream)
        for _ in range(Ke):
            e2e_run()
        eb.record(stream)
        barrier()
        ems = all_reduce_scalar(ea.elapsed_time(eb) / Ke, "max", dev)
        e2e = {"value": whole_job_rate(T, world, ems), "unit": "tokens/s",
               "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in host_in),
               "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in host_dp),
               "ms_per_step": ems, "steps": Ke,
               "pipeline": "inputs in and dparams out every step, in stream order"}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        small = synth.draw_encoder(256, seed=0)
        encoder_oracle_step(small)
        n, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < 10.0:
            encoder_oracle_step(small)
            n += 1
        el = time.perf_counter() - t0
        cpu = {"value": n * 256 / el, "unit": "tokens/s", "cores": oracle_threads(),
               "kind": "oracle", "cpu_model": cpu_model(), "nproc": os.cpu_count(),
               "sample": f"{n} block steps of the fp64 numpy oracle on 256 of the {T} tokens "
                         f"({el:.1f} s)"}
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "timing": dict(rep, note="ms_per_step is the median over repeats of the K-step "
                                     "region, max over ranks"),
            "config": {"workload": "encoder768_bf16",
                       "description": "the TT layers of one encoder block: Q, K, V, O "
                                      "(768x768, ranks 30) and the GELU FFN pair "
                                      "768->3072->768, fwd+bwd of all, 16384 tokens, bf16",
                       "tokens": T, "parallelism": f"replicas x{world}", "launch": note,
                       "deterministic": bool(args.deterministic),
                       "qkv": "separate plans" if args.no_fuse_qkv else "one multi-layer plan",
                       "l2": f"{nsets} rotating input sets of {set_bytes / 1e6:.0f} MB"},
            "roofline": {"bound": "hbm", "kernel": "whole block step (summed)",
                         "achieved": byts / (ms * 1e-3) / 1e9, "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": t_roof / (ms * 1e-3), "traffic": None,
                         "algorithmic_bytes_per_step": byts},
            "roofline_step": {"t_roof_us": t_roof * 1e6, "frac": t_roof / (ms * 1e-3),
                              "algorithmic_bytes": byts, "algorithmic_flop": flop,
                              "peak_gbs": peak, "peak_kind": peak_kind},
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse()
    if args.oracle_rate:
        oracle_rate_main(args)
        return
    from tensor_train_compressed_tt_gb300 import synth
    if args.workload in synth.TTM_WORKLOADS:
        w = synth.TTM_WORKLOADS[args.workload]
        if args.impl == "reference":
            run_ttm_reference(args, w)
        else:
            run_ttm(args, w)
        return
    if args.workload == "encoder768_bf16":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the reference arm times single workloads; use --workload"}))
        else:
            run_encoder(args)
        return
    w = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
