#!/usr/bin/env python
"""Benchmark of the AdaLN norm_out forward + backward on GB300.

One step = the whole hot path on one batch of synthetic inputs already in
HBM: adaln_proj_fwd, adaln_out_fwd, adaln_out_bwd, adaln_proj_bwd (bf16 dW,
db) at B=2, S=4096, D=3072 with 1% outlier rows.  The headline is tokens/s;
the JSON line also carries HBM GB/s from the algorithmic bytes, the roofline
of the dominant call, an end-to-end number through host buffers, the CPU
oracle's throughput and the SM clocks seen during the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
    python bench.py --proj-sweep      # the projection calls alone, B = 1 .. 2048

Under torchrun (N > 1) every rank runs its own replica (weak scaling; the
path has no cross-sample exchange), the elapsed time is the max over ranks
and rank 0 prints one JSON line.  --impl reference runs the CPU oracle on a
bounded sample of the same workload (rank 0 only).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "AdaLN-out fwd+bwd tokens/s and HBM GB/s (% of 8 TB/s) at B=2,S=4096,D=3072"
WORKLOAD = dict(B=2, S=4096, D=3072, seed=0, outlier_frac=0.01)
NOMINAL_HBM_GBS = 8000.0
FLUSH_BYTES = 512 << 20
KERNELS_PER_STEP = 7  # SiLU, projection, out_fwd, bwd tile, tree fold, proj-bwd slab, d_temb
# DRAM bytes (read + write) of one adaln_out_bwd call (tile kernel + tree fold) at this
# workload, from the ncu capture summarised in profiles/out_bwd_B2_S4096_D3072.md.  The
# counters of a replayed launch miss the dx lines still in L2 when it ends.
OUT_BWD_DRAM_BYTES = 133_192_704


# ---------------------------------------------------------------------------
# algorithmic bytes (what the method must move; workspaces excluded)
# ---------------------------------------------------------------------------

def call_bytes(B, S, D):
    """Bytes each C-ABI call must read and write once, by tensor sizes."""
    N = 2 * D
    rows = B * S
    bf, f4 = 2, 4
    return {
        "adaln_proj_fwd": B * D * bf + N * D * bf + N * bf + B * N * bf + B * D * bf,
        "adaln_out_fwd": rows * D * bf + B * N * bf + rows * D * bf + 2 * rows * f4,
        "adaln_out_bwd": 2 * rows * D * bf + B * N * bf + 2 * rows * f4 + rows * D * bf + B * N * f4,
        "adaln_proj_bwd": B * N * f4 + 2 * B * D * bf + N * D * bf + B * D * bf + N * D * bf + N * bf,
    }


def step_bytes(B, S, D):
    return sum(call_bytes(B, S, D).values())


# ---------------------------------------------------------------------------
# distributed plumbing (host side; also exercised on CPU with gloo)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist_mod, device=None):
    if dist_mod is not None:
        if device is not None:
            dist_mod.barrier(device_ids=[device.index])
        else:
            dist_mod.barrier()


def max_over_ranks(value: float, dist_mod, device=None) -> float:
    if dist_mod is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device if device is not None else "cpu")
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    return float(t.item())


def throughput(units_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job throughput: the units all ranks processed over the max time."""
    return units_per_rank * world / seconds


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        return summarize_clocks(self.lines)


def summarize_clocks(lines):
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for ln in lines:
        parts = [p.strip() for p in ln.split(",")]
        if len(parts) < 8:
            continue
        try:
            sm.append(float(parts[0]))
            mx.append(float(parts[1]))
        except ValueError:
            continue
        for name, val in zip(names, parts[4:8]):
            if val.lower().startswith("active"):
                reasons.add(name)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
            "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle timing (a bounded sample of the workload)
# ---------------------------------------------------------------------------

def oracle_sample_step(oracle, inp, frac, emb_full=None):
    """The oracle's chain on a fraction `frac` of the workload, so that every
    stage does `frac` of its full work: the projection forward and backward on
    the first frac*2D output rows, the LayerNorm forward and backward on the
    first frac*S tokens of every sample (with the full emb).  frac = 1 is the
    whole workload through the oracle's full entry points.  Returns seconds."""
    B, S, D = inp["x"].shape
    t0 = time.perf_counter()
    if frac >= 1:
        emb = oracle.proj_fwd(inp["temb"], inp["W"], inp["b"])
        _, _, _ = oracle.out_fwd(inp["x"], emb)
        _, d_emb = oracle.out_bwd(inp["dy"], inp["x"], emb)
        oracle.proj_bwd(d_emb, inp["temb"], inp["W"])
        return time.perf_counter() - t0
    s = max(1, int(round(S * frac)))
    n = max(1, int(round(2 * D * frac)))
    oracle.proj_fwd_rows(inp["temb"], inp["W"], inp["b"], 0, n, emb=emb_full.copy())
    x = np.ascontiguousarray(inp["x"][:, :s])
    dy = np.ascontiguousarray(inp["dy"][:, :s])
    oracle.out_fwd(x, emb_full)
    _, d_emb = oracle.out_bwd(dy, x, emb_full)
    oracle.proj_bwd_rows(d_emb, inp["temb"], inp["W"], 0, n)
    return time.perf_counter() - t0


def time_oracle(inp, budget_s=12.0, max_steps=50):
    """Run the full oracle chain repeatedly for about budget_s seconds."""
    import oracle
    oracle.build()
    B, S, _ = inp["x"].shape
    times = []
    t_start = time.perf_counter()
    while not times or (time.perf_counter() - t_start < budget_s and len(times) < max_steps):
        times.append(oracle_sample_step(oracle, inp, 1.0))
    total = sum(times)
    return {"value": B * S * len(times) / total, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{len(times)} full steps of B={B}, S={S} (all tokens, all projection rows), single thread",
            "seconds": total}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

def run_gpu(args, world, rank, local):
    import torch
    from invariant_dit_adaln_gb300 import binding, build, synth

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist_mod = init_dist(world, "nccl")
    # one rank builds (a no-op when the library is up to date); the others wait
    # for it rather than compile into the same files at the same time
    if rank == 0:
        build.build()
    barrier(dist_mod, device)
    binding.load()

    W_ = WORKLOAD
    B, S, D = W_["B"], W_["S"], W_["D"]
    N = 2 * D
    host = synth.make_inputs(B, S, D, seed=W_["seed"] + rank, outlier_frac=W_["outlier_frac"])

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)

    x, dy, temb, W, b = (dev(host[k]) for k in ("x", "dy", "temb", "W", "b"))
    emb = torch.empty((B, N), dtype=torch.bfloat16, device=device)
    u = torch.empty((B, D), dtype=torch.bfloat16, device=device)
    out = torch.empty((B, S, D), dtype=torch.bfloat16, device=device)
    mean = torch.empty((B, S), dtype=torch.float32, device=device)
    rstd = torch.empty((B, S), dtype=torch.float32, device=device)
    dx = torch.empty_like(out)
    d_emb = torch.empty((B, N), dtype=torch.float32, device=device)
    d_temb = torch.empty((B, D), dtype=torch.bfloat16, device=device)
    dW = torch.empty((N, D), dtype=torch.bfloat16, device=device)
    db = torch.empty((N,), dtype=torch.bfloat16, device=device)
    ws_bwd = torch.empty(binding.adaln_out_bwd_workspace_bytes(B, S, D), dtype=torch.uint8, device=device)
    ws_proj = torch.empty(binding.adaln_proj_bwd_workspace_bytes(B, D), dtype=torch.uint8, device=device)
    flush_w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    flush_r = torch.zeros(FLUSH_BYTES // 4, dtype=torch.int32, device=device)

    def flush():
        # Between steps, outside the timed events: write a buffer 4x the L2
        # (no line of the step's inputs or outputs stays cached), then read
        # another one, so the dirty lines of the write are written back here
        # rather than inside the next step.
        flush_w.zero_()
        flush_r.max()
    stream = torch.cuda.current_stream(device)

    def step(st=stream):
        binding.adaln_proj_fwd(temb, W, b, emb=emb, u=u, stream=st)
        binding.adaln_out_fwd(x, emb, out=out, mean=mean, rstd=rstd, stream=st)
        binding.adaln_out_bwd(dy, x, emb, mean, rstd, dx=dx, d_emb=d_emb, workspace=ws_bwd, stream=st)
        binding.adaln_proj_bwd(d_emb, temb, u, W, d_temb=d_temb, dW=dW, db=db, workspace=ws_proj, stream=st)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    assert binding.device_error() == 0

    # The step's seven launches captured once in a CUDA graph (after the
    # warm-up, which also filled the SiLU table); the programmatic dependent
    # launch edges between the kernels are kept.  The timed loop replays it.
    graph = None
    if not args.eager:
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(device)
        cap.wait_stream(stream)
        with torch.cuda.graph(graph, stream=cap):
            step(torch.cuda.current_stream(device))
        torch.cuda.synchronize()
        assert binding.device_error() == 0

    def run_step():
        if graph is not None:
            graph.replay()
        else:
            step()

    # ---- timed region: K steps, per-step events, L2 flushed between steps ----
    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    clocks = ClockSampler(local)
    barrier(dist_mod, device)
    torch.cuda.synchronize()
    clocks.start()
    wall0 = time.perf_counter()
    for i in range(K):
        flush()
        starts[i].record(stream)
        run_step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    barrier(dist_mod, device)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    my_time = sum(step_ms) / 1e3
    t_max = max_over_ranks(my_time, dist_mod, device)
    assert binding.device_error() == 0

    # the same steps launched one call at a time, for comparison
    K1 = min(K, 300)
    eg = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K1)]
    for i in range(K1):
        flush()
        eg[i][0].record(stream)
        step()
        eg[i][1].record(stream)
    torch.cuda.synchronize()
    eager_ms = statistics.mean(a.elapsed_time(c) for a, c in eg)

    # ---- per-call pass: events around each call (roofline of the dominant call) ----
    K2 = min(K, 300)
    names = ["adaln_proj_fwd", "adaln_out_fwd", "adaln_out_bwd", "adaln_proj_bwd"]
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K2)]
    calls = [
        lambda: binding.adaln_proj_fwd(temb, W, b, emb=emb, u=u, stream=stream),
        lambda: binding.adaln_out_fwd(x, emb, out=out, mean=mean, rstd=rstd, stream=stream),
        lambda: binding.adaln_out_bwd(dy, x, emb, mean, rstd, dx=dx, d_emb=d_emb, workspace=ws_bwd, stream=stream),
        lambda: binding.adaln_proj_bwd(d_emb, temb, u, W, d_temb=d_temb, dW=dW, db=db, workspace=ws_proj,
                                       stream=stream),
    ]
    for i in range(K2):
        flush()
        ev[i][0].record(stream)
        for j, c in enumerate(calls):
            c()
            ev[i][j + 1].record(stream)
    torch.cuda.synchronize()
    call_ms = {n: statistics.mean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(K2)) for j, n in enumerate(names)}

    # ---- end to end: host buffers in, host buffers out, every step ----
    K3 = min(K, 100)
    pin = {k: torch.from_numpy(np.ascontiguousarray(host[k]).view(np.int16)).view(torch.bfloat16).pin_memory()
           for k in ("x", "dy", "temb", "W", "b")}
    outs_h = {"out": torch.empty(out.shape, dtype=out.dtype).pin_memory(),
              "dx": torch.empty(dx.shape, dtype=dx.dtype).pin_memory(),
              "emb": torch.empty(emb.shape, dtype=emb.dtype).pin_memory(),
              "d_emb": torch.empty(d_emb.shape, dtype=d_emb.dtype).pin_memory(),
              "d_temb": torch.empty(d_temb.shape, dtype=d_temb.dtype).pin_memory(),
              "dW": torch.empty(dW.shape, dtype=dW.dtype).pin_memory(),
              "db": torch.empty(db.shape, dtype=db.dtype).pin_memory()}
    dev_out = {"out": out, "dx": dx, "emb": emb, "d_emb": d_emb, "d_temb": d_temb, "dW": dW, "db": db}
    dev_in = {"x": x, "dy": dy, "temb": temb, "W": W, "b": b}
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = sum(t.numel() * t.element_size() for t in outs_h.values())
    # A stream of steps, each with its own host inputs copied in and its results
    # copied out, pipelined over two sets of device buffers: step i + 1's inputs
    # go in (one stream, in the order the calls need them) while step i computes
    # (the compute stream) and its results come out (a third stream, each tensor
    # as soon as the call that writes it is done).  A set is reused only after
    # the step two back has finished reading its inputs and its results are out.
    # No L2 flush: each step's 138 MB of inputs exceeds L2.  The timed region runs
    # from before the first copy in to after the last copy out.
    s_in = torch.cuda.Stream(device)
    s_out = torch.cuda.Stream(device)

    def dev_set():
        d = {k: torch.empty_like(v) for k, v in dev_in.items()}
        d.update({k: torch.empty_like(v) for k, v in dev_out.items()})
        d["u"] = torch.empty_like(u)
        d["mean"] = torch.empty_like(mean)
        d["rstd"] = torch.empty_like(rstd)
        d["ws_bwd"] = torch.empty_like(ws_bwd)
        d["ws_proj"] = torch.empty_like(ws_proj)
        return d

    sets = [dev_set(), dev_set()]

    def ev(st):
        e = torch.cuda.Event()
        e.record(st)
        return e

    free_in = [None, None]   # event: the set's inputs are no longer read
    free_out = [None, None]  # event: the set's results have been copied out
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    stream.wait_event(t0)
    s_out.wait_event(t0)
    for i in range(K3):
        d = sets[i % 2]
        if free_in[i % 2] is not None:
            s_in.wait_event(free_in[i % 2])
        with torch.cuda.stream(s_in):
            for k in ("temb", "W", "b"):
                d[k].copy_(pin[k], non_blocking=True)
            e_proj = ev(s_in)
            d["x"].copy_(pin["x"], non_blocking=True)
            e_x = ev(s_in)
            d["dy"].copy_(pin["dy"], non_blocking=True)
            e_dy = ev(s_in)
        if free_out[i % 2] is not None:
            stream.wait_event(free_out[i % 2])
        stream.wait_event(e_proj)
        binding.adaln_proj_fwd(d["temb"], d["W"], d["b"], emb=d["emb"], u=d["u"], stream=stream)
        stream.wait_event(e_x)
        binding.adaln_out_fwd(d["x"], d["emb"], out=d["out"], mean=d["mean"], rstd=d["rstd"], stream=stream)
        e_fwd = ev(stream)
        stream.wait_event(e_dy)
        binding.adaln_out_bwd(d["dy"], d["x"], d["emb"], d["mean"], d["rstd"], dx=d["dx"], d_emb=d["d_emb"],
                              workspace=d["ws_bwd"], stream=stream)
        e_bwd = ev(stream)
        binding.adaln_proj_bwd(d["d_emb"], d["temb"], d["u"], d["W"], d_temb=d["d_temb"], dW=d["dW"], db=d["db"],
                               workspace=d["ws_proj"], stream=stream)
        e_end = ev(stream)
        free_in[i % 2] = e_end
        with torch.cuda.stream(s_out):
            s_out.wait_event(e_fwd)
            for k in ("out", "emb"):
                outs_h[k].copy_(d[k], non_blocking=True)
            s_out.wait_event(e_bwd)
            for k in ("dx", "d_emb"):
                outs_h[k].copy_(d[k], non_blocking=True)
            s_out.wait_event(e_end)
            for k in ("d_temb", "dW", "db"):
                outs_h[k].copy_(d[k], non_blocking=True)
            free_out[i % 2] = ev(s_out)
    t1.record(s_out)
    torch.cuda.synchronize()
    e2e_s = t0.elapsed_time(t1) / 1e3
    # the last step's results equal the ones computed in place
    assert torch.equal(outs_h["dW"].view(torch.int16), dW.cpu().view(torch.int16))
    e2e_max = max_over_ranks(e2e_s, dist_mod, device)
    assert binding.device_error() == 0

    tokens = B * S
    value = throughput(tokens * K, world, t_max)
    sbytes = step_bytes(B, S, D)
    gbs = sbytes * K / my_time / 1e9
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except OSError:
        pass
    peak = float(peaks.get("hbm_gbs", 6800.0))
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    cb = call_bytes(B, S, D)
    dom = "adaln_out_bwd"
    ach = cb[dom] / (call_ms[dom] / 1e3) / 1e9
    result = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": my_time / K * 1e3,
        "ms_per_step_eager": eager_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "compute": "fp32 arithmetic on bf16 tensors",
        "data": "synthetic (seeded; x, dy ~ N(0,1) with 81 outlier rows x50; W, b ~ N(0, 0.02^2))",
        "config": {"workload": "AdaLN norm_out fwd+bwd, B=2 S=4096 D=3072, 1% outlier rows",
                   "B": B, "S": S, "D": D, "parallelism": "replicas" if world > 1 else "single GPU",
                   "launch": ("eager: one C-ABI call at a time" if graph is None else
                              "CUDA graph of the step's four C-ABI calls (7 kernels, programmatic launch edges), "
                              "captured once after the warm-up and replayed each step"),
                   "l2": "flushed between steps outside the timed events: 512 MiB write, then 512 MiB read (L2 cold and clean at each step start); inputs 138 MB > L2"},
        "hbm_gbs": gbs,
        "hbm_frac_of_8tbs": gbs / NOMINAL_HBM_GBS,
        "hbm_frac_of_measured": gbs / peak,
        "algorithmic_bytes_per_step": sbytes,
        "calls_ms": call_ms,
        "roofline": {"bound": "hbm", "kernel": dom + " (LN-backward tile kernel + tree fold)",
                     "achieved": ach, "peak": peak, "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)",
                     "unit": "GB/s", "frac": ach / peak, "traffic": OUT_BWD_DRAM_BYTES,
                     "algorithmic_bytes": cb[dom]},
        "step_roofline": {"achieved": gbs, "peak": peak, "frac": gbs / peak, "unit": "GB/s"},
        "e2e": {"value": throughput(tokens * K3, world, e2e_max), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": KERNELS_PER_STEP * K,
        "clocks": clk,
        "wall_s": wall,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = time_oracle(host, budget_s=args.cpu_budget)
    if dist_mod is not None:
        dist_mod.destroy_process_group()
    return result if rank == 0 else None


# ---------------------------------------------------------------------------
# the reference arm: the CPU oracle on the same workload
# ---------------------------------------------------------------------------

def run_reference(args, world, rank):
    if rank != 0:
        return None
    import oracle
    from invariant_dit_adaln_gb300 import synth
    oracle.build()
    W_ = WORKLOAD
    B, S, D = W_["B"], W_["S"], W_["D"]
    inp = synth.make_inputs(B, S, D, seed=W_["seed"], outlier_frac=W_["outlier_frac"])
    # size the sample so that warmup + steps take about args.ref_budget seconds
    emb_full = oracle.proj_fwd(inp["temb"], inp["W"], inp["b"])
    t_cal = oracle_sample_step(oracle, inp, 1.0 / 64, emb_full)
    per_step = args.ref_budget / max(1, args.steps + args.warmup)
    frac = min(1.0, max(1.0 / 1024, (1.0 / 64) * per_step / max(t_cal, 1e-6)))
    frac = float(2.0 ** np.floor(np.log2(frac)))
    for _ in range(args.warmup):
        oracle_sample_step(oracle, inp, frac, emb_full)
    times = [oracle_sample_step(oracle, inp, frac, emb_full) for _ in range(args.steps)]
    total = sum(times)
    tokens = B * S * frac * len(times)
    value = tokens / total
    part = "the whole workload" if frac >= 1.0 else f"a fraction {frac:g} of the workload"
    sample = (f"each step: the oracle chain on {part} (first {max(1, int(round(S * frac)))} "
              f"tokens of each of B={B} samples, {max(1, int(round(2 * D * frac)))} of {2 * D} projection rows), "
              f"single thread")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total / len(times) * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64 (oracle; bf16 rounding points emulated)",
        "data": "synthetic (seeded; same inputs as the GPU arm)",
        "config": {"workload": "AdaLN norm_out fwd+bwd, B=2 S=4096 D=3072, 1% outlier rows",
                   "B": B, "S": S, "D": D, "parallelism": "CPU, rank 0 only"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_proj_sweep(args, rank, local):
    """The two projection calls alone over the conditioning batch B (D = 3072,
    weights N(0, 0.02^2)): each call timed by CUDA events on its stream, the
    median of several runs, L2 flushed before each.  One JSON line per B, on
    rank 0; a diagnostic of how the CUDA-core projections grow with B, not
    the headline."""
    if rank != 0:
        return
    import torch
    from invariant_dit_adaln_gb300 import binding, build, synth

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    build.build()
    binding.load()
    D = WORKLOAD["D"]
    N = 2 * D
    host = synth.make_inputs(2048, 1, D, seed=WORKLOAD["seed"])

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)

    W, b, temb_all = dev(host["W"]), dev(host["b"]), dev(host["temb"])
    d_emb_all = torch.from_numpy(synth.normal(synth.stream_key(WORKLOAD["seed"], "aux"), 2048 * N)
                                 .astype(np.float32).reshape(2048, N)).to(device)
    dW = torch.empty((N, D), dtype=torch.bfloat16, device=device)
    db = torch.empty((N,), dtype=torch.bfloat16, device=device)
    flush_w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    st = torch.cuda.current_stream(device)
    for B in [1, 2, 8, 64, 257, 2048]:
        temb, d_emb = temb_all[:B].contiguous(), d_emb_all[:B].contiguous()
        emb = torch.empty((B, N), dtype=torch.bfloat16, device=device)
        u = torch.empty((B, D), dtype=torch.bfloat16, device=device)
        d_temb = torch.empty((B, D), dtype=torch.bfloat16, device=device)
        ws = torch.empty(max(1, binding.adaln_proj_bwd_workspace_bytes(B, D)), dtype=torch.uint8, device=device)
        calls = {"adaln_proj_fwd": lambda: binding.adaln_proj_fwd(temb, W, b, emb=emb, u=u, stream=st),
                 "adaln_proj_bwd": lambda: binding.adaln_proj_bwd(d_emb, temb, u, W, d_temb=d_temb, dW=dW, db=db,
                                                                  workspace=ws, stream=st)}
        runs = 20 if B >= 257 else 100
        res = {}
        for name, call in calls.items():
            call()
            torch.cuda.synchronize(device)
            ts = []
            for _ in range(runs):
                flush_w.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(st)
                call()
                e1.record(st)
                torch.cuda.synchronize(device)
                ts.append(e0.elapsed_time(e1) * 1e3)
            res[name] = statistics.median(ts)
        if binding.device_error() != 0:
            raise RuntimeError("device-side error during the projection sweep")
        flops = {"adaln_proj_fwd": 2.0 * B * N * D, "adaln_proj_bwd": 4.0 * B * N * D}
        print(json.dumps({"sweep": "projections", "B": B, "D": D, "us": res,
                          "tflops": {k: flops[k] / (v * 1e-6) / 1e12 for k, v in res.items()},
                          "runs": runs, "l2": "512 MiB write before each run"}), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=90.0, help="seconds for the reference arm's steps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true", help="time the step as separate calls, not a CUDA graph")
    ap.add_argument("--proj-sweep", action="store_true",
                    help="instead of the step: time the projection calls alone for B = 1 .. 2048")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_env()
    if args.proj_sweep:
        run_proj_sweep(args, rank, local)
        return
    if args.impl == "reference":
        res = run_reference(args, world, rank)
    else:
        res = run_gpu(args, world, rank, local)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
