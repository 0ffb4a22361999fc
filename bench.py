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
    python bench.py --chunking        # 4096 samples of S=256 in five chunkings

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
# kernels per step at this workload: SiLU, tensor-core projection, LayerNorm
# forward, backward tile, tree fold, projection-backward slab, d_temb
KERNELS_PER_STEP = 7
# DRAM bytes (read + write) of one adaln_out_bwd call (tile kernel + tree fold)
# at this workload, from one ncu capture of the current kernels
# (dram__bytes_read.sum + dram__bytes_write.sum of both kernels, mean of two
# calls; dx lines still in L2 when a replayed launch ends are not counted).
# None when the kernels change after the capture.
OUT_BWD_DRAM_BYTES = 117_004_800


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

class NvmlSampler:
    """SM clock, max clock, power and clock-event reasons of one GPU, read
    through NVML every `period_s` seconds in a thread (reads only; no setting is
    changed).  Each sample carries its time, so samples can be binned by pass."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, pci_bus_id=None, index=0, period_s=0.005):
        import ctypes
        self.period = period_s
        self.samples = []  # (t, sm_mhz, max_mhz, power_w, reasons bitmask)
        self._stop = threading.Event()
        L = ctypes.CDLL("libnvidia-ml.so.1")
        if L.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.L = L
        self.h = ctypes.c_void_p()
        rc = 1
        if pci_bus_id:
            rc = L.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(self.h))
        if rc != 0:
            rc = L.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h))
        if rc != 0:
            raise OSError("no NVML handle")
        self.c = ctypes

    def _read(self):
        c, L = self.c, self.L
        sm, mx, pw, rs = c.c_uint(), c.c_uint(), c.c_uint(), c.c_ulonglong()
        L.nvmlDeviceGetClockInfo(self.h, 1, c.byref(sm))        # NVML_CLOCK_SM
        L.nvmlDeviceGetMaxClockInfo(self.h, 1, c.byref(mx))
        L.nvmlDeviceGetPowerUsage(self.h, c.byref(pw))
        (getattr(L, "nvmlDeviceGetCurrentClocksEventReasons", None) or
         L.nvmlDeviceGetCurrentClocksThrottleReasons)(self.h, c.byref(rs))
        return (time.perf_counter(), float(sm.value), float(mx.value), pw.value / 1000.0, int(rs.value))

    def _run(self):
        while not self._stop.is_set():
            self.samples.append(self._read())
            time.sleep(self.period)

    def start(self):
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def stop(self):
        self._stop.set()
        self.thread.join(timeout=5)

    def summary(self, windows=None):
        """Median SM clock etc. over the samples inside the (t0, t1) windows."""
        sel = [x for x in self.samples if windows is None or any(a <= x[0] <= b for a, b in windows)]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0, "source": "nvml"}
        mask = 0
        for x in sel:
            mask |= x[4]
        return {"sm_mhz": statistics.median(x[1] for x in sel), "sm_max_mhz": max(x[2] for x in sel),
                "power_w_max": max(x[3] for x in sel),
                "reasons": sorted(n for bit, n in self.REASONS.items() if mask & bit), "samples": len(sel),
                "source": "nvml"}


class ClockSampler:
    """Fallback when NVML cannot be loaded: nvidia-smi every 20 ms."""
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
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)

    def summary(self, windows=None):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        r = summarize_clocks(self.lines)
        r["source"] = "nvidia-smi"
        return r


def clock_sampler(device_index):
    """NVML sampler for the CUDA device (matched by PCI bus id), else nvidia-smi."""
    bus = None
    try:
        import torch
        pr = torch.cuda.get_device_properties(device_index)
        if hasattr(pr, "pci_bus_id"):
            bus = f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0"
    except Exception:
        bus = None
    try:
        return NvmlSampler(pci_bus_id=bus, index=device_index)
    except OSError:
        return ClockSampler(device_index)


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


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


_SHARED = {}


def _pool_init(specs):
    """Worker start-up: attach to the inputs in shared memory, load the oracle."""
    from multiprocessing import shared_memory
    import oracle
    oracle.build()
    for k, (name, shape, dtype) in specs.items():
        shm = shared_memory.SharedMemory(name=name)
        _SHARED[k] = (shm, np.ndarray(shape, dtype=dtype, buffer=shm.buf))


def _pool_share(args):
    """One worker's share of the oracle step: its tokens [s0, s1) of every
    sample through the LayerNorm forward and backward, and its projection rows
    [n0, n1) forward and backward.  Returns its seconds."""
    i, P = args
    import oracle
    x, dy, temb, W, b, emb = (_SHARED[k][1] for k in ("x", "dy", "temb", "W", "b", "emb"))
    B, S, D = x.shape
    s0, s1 = S * i // P, S * (i + 1) // P
    n0, n1 = 2 * D * i // P, 2 * D * (i + 1) // P
    t0 = time.perf_counter()
    oracle.proj_fwd_rows(temb, W, b, n0, n1, emb=emb.copy())
    xs, dys = np.ascontiguousarray(x[:, s0:s1]), np.ascontiguousarray(dy[:, s0:s1])
    oracle.out_fwd(xs, emb)
    _, d_emb = oracle.out_bwd(dys, xs, emb)
    oracle.proj_bwd_rows(d_emb, temb, W, n0, n1)
    return time.perf_counter() - t0


def time_oracle(inp, budget_s=12.0, max_steps=50):
    """The oracle as it stands on the host: full steps on one thread for about
    budget_s / 3 seconds, then whole steps split over every host core (spawned
    worker processes, each running the oracle chain on its own share of the
    tokens and projection rows) for about 2 budget_s / 3 seconds."""
    import multiprocessing as mp
    from multiprocessing import shared_memory
    import oracle
    oracle.build()
    B, S, D = inp["x"].shape
    times = []
    t_start = time.perf_counter()
    while not times or (time.perf_counter() - t_start < budget_s / 3 and len(times) < max_steps):
        times.append(oracle_sample_step(oracle, inp, 1.0))
    single = B * S * len(times) / sum(times)
    emb = oracle.proj_fwd(inp["temb"], inp["W"], inp["b"])
    arrays = {"x": inp["x"], "dy": inp["dy"], "temb": inp["temb"], "W": inp["W"], "b": inp["b"], "emb": emb}
    P = os.cpu_count() or 1
    shms, specs = [], {}
    try:
        for k, a in arrays.items():
            a = np.ascontiguousarray(a)
            shm = shared_memory.SharedMemory(create=True, size=max(1, a.nbytes))
            np.ndarray(a.shape, dtype=a.dtype, buffer=shm.buf)[...] = a
            shms.append(shm)
            specs[k] = (shm.name, a.shape, a.dtype.str)
        walls = []
        with mp.get_context("spawn").Pool(P, initializer=_pool_init, initargs=(specs,)) as pool:
            # every map has a time limit: a pool whose workers cannot start would
            # otherwise wait forever
            limit = 10 * budget_s + 60
            pool.map_async(_pool_share, [(i, P) for i in range(P)]).get(timeout=limit)  # warm-up
            t_start = time.perf_counter()
            while not walls or (time.perf_counter() - t_start < 2 * budget_s / 3 and len(walls) < max_steps):
                w0 = time.perf_counter()
                pool.map_async(_pool_share, [(i, P) for i in range(P)]).get(timeout=limit)
                walls.append(time.perf_counter() - w0)
    except (mp.TimeoutError, OSError) as e:
        return {"value": single, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                "sample": f"{len(times)} full steps of B={B}, S={S}, single thread (the multi-process run failed: {e!r})",
                "single_thread_value": single, "cpu_model": cpu_model(), "nproc": P}
    finally:
        for shm in shms:
            shm.close()
            shm.unlink()
    value = B * S * len(walls) / sum(walls)
    return {"value": value, "unit": "tokens/s", "cores": P, "kind": "oracle",
            "sample": (f"{len(walls)} full steps of B={B}, S={S}, each split over {P} worker processes "
                       f"(tokens and projection rows in {P} shares); single thread: {len(times)} full steps"),
            "single_thread_value": single, "cpu_model": cpu_model(), "nproc": P, "seconds": sum(walls)}


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

    def make_set():
        """The step's inputs (the same seeded values), outputs and workspaces in
        buffers of their own: 138 MB of inputs per set, more than L2 holds."""
        d = {k: dev(host[k]) for k in ("x", "dy", "temb", "W", "b")}
        d.update(emb=torch.empty((B, N), dtype=torch.bfloat16, device=device),
                 u=torch.empty((B, D), dtype=torch.bfloat16, device=device),
                 out=torch.empty((B, S, D), dtype=torch.bfloat16, device=device),
                 mean=torch.empty((B, S), dtype=torch.float32, device=device),
                 rstd=torch.empty((B, S), dtype=torch.float32, device=device),
                 dx=torch.empty((B, S, D), dtype=torch.bfloat16, device=device),
                 d_emb=torch.empty((B, N), dtype=torch.float32, device=device),
                 d_temb=torch.empty((B, D), dtype=torch.bfloat16, device=device),
                 dW=torch.empty((N, D), dtype=torch.bfloat16, device=device),
                 db=torch.empty((N,), dtype=torch.bfloat16, device=device),
                 ws_bwd=torch.empty(binding.adaln_out_bwd_workspace_bytes(B, S, D), dtype=torch.uint8, device=device),
                 ws_proj=torch.empty(binding.adaln_proj_bwd_workspace_bytes(B, D), dtype=torch.uint8, device=device))
        return d

    sets = [make_set(), make_set()]
    A = sets[0]
    x, dy, temb, W, b = A["x"], A["dy"], A["temb"], A["W"], A["b"]
    emb, u, out, mean, rstd, dx = A["emb"], A["u"], A["out"], A["mean"], A["rstd"], A["dx"]
    d_emb, d_temb, dW, db, ws_bwd, ws_proj = A["d_emb"], A["d_temb"], A["dW"], A["db"], A["ws_bwd"], A["ws_proj"]
    flush_w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    flush_r = torch.zeros(FLUSH_BYTES // 4, dtype=torch.int32, device=device)

    def flush():
        # Between steps of the flushed pass, outside its timed events: write a
        # buffer 4x the L2 (no line of the step's inputs or outputs stays
        # cached), then read another one, so the dirty lines of the write are
        # written back here rather than inside the next step.
        flush_w.zero_()
        flush_r.max()
    stream = torch.cuda.current_stream(device)

    def step_on(d, st=stream):
        binding.adaln_proj_fwd(d["temb"], d["W"], d["b"], emb=d["emb"], u=d["u"], stream=st)
        binding.adaln_out_fwd(d["x"], d["emb"], out=d["out"], mean=d["mean"], rstd=d["rstd"], stream=st)
        binding.adaln_out_bwd(d["dy"], d["x"], d["emb"], d["mean"], d["rstd"], dx=d["dx"], d_emb=d["d_emb"],
                              workspace=d["ws_bwd"], stream=st)
        binding.adaln_proj_bwd(d["d_emb"], d["temb"], d["u"], d["W"], d_temb=d["d_temb"], dW=d["dW"], db=d["db"],
                               workspace=d["ws_proj"], stream=st)

    def step(st=stream):
        step_on(A, st)

    for i in range(args.warmup):
        step_on(sets[i % 2])
    torch.cuda.synchronize()
    assert binding.device_error() == 0

    # The step's launches captured once per input set in a CUDA graph (after the
    # warm-up, which also filled the SiLU table); the programmatic dependent
    # launch edges between the kernels are kept.  The timed loops replay them.
    graphs = None
    if not args.eager:
        graphs = []
        cap = torch.cuda.Stream(device)
        cap.wait_stream(stream)
        for d in sets:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                step_on(d, torch.cuda.current_stream(device))
            graphs.append(g)
        torch.cuda.synchronize()
        assert binding.device_error() == 0

    def run_step(i):
        if graphs is not None:
            graphs[i % 2].replay()
        else:
            step_on(sets[i % 2])

    # ---- timed region: passes of exactly K steps back to back ----
    # Consecutive steps alternate between the two input sets, each larger than
    # L2, so no step finds its inputs cached by the step before.  One event pair
    # on the launch stream brackets the K steps of a pass, with a barrier and a
    # synchronize on both sides.  Passes repeat until about --min-timed-s
    # seconds have been timed (the clocks are sampled throughout); the pass with
    # the median time is reported, all passes are listed.
    K = args.steps
    clocks = clock_sampler(local)
    clocks.start()
    passes, windows = [], []
    t_begin = time.perf_counter()
    while len(passes) < 3 or (time.perf_counter() - t_begin < args.min_timed_s and len(passes) < args.max_passes):
        barrier(dist_mod, device)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        w0 = time.perf_counter()
        e0.record(stream)
        for i in range(K):
            run_step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        windows.append((w0, time.perf_counter()))
        barrier(dist_mod, device)
        passes.append(e0.elapsed_time(e1) / 1e3)
    wall = time.perf_counter() - t_begin
    clocks.stop()
    clk = clocks.summary(windows)
    my_time = statistics.median(passes)
    t_max = max_over_ranks(my_time, dist_mod, device)
    assert binding.device_error() == 0
    # the passes in ten consecutive bins: each bin's median time per step next to
    # the median SM clock sampled over its span, and their product, so that any
    # dependence on the clock shows
    bins = []
    nb = min(10, len(passes))
    for k in range(nb):
        lo, hi = k * len(passes) // nb, (k + 1) * len(passes) // nb
        ms = statistics.median(passes[lo:hi]) / K * 1e3
        mhz = clocks.summary([(windows[lo][0], windows[hi - 1][1])]).get("sm_mhz")
        bins.append({"passes": hi - lo, "ms_per_step": ms, "sm_mhz": mhz,
                     "ms_x_mhz": ms * mhz if mhz else None})

    # ---- the same steps with the L2 flushed between them, one event pair per step ----
    K1 = min(K, 300)
    fl = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K1)]
    for i in range(K1):
        flush()
        fl[i][0].record(stream)
        run_step(0)
        fl[i][1].record(stream)
    torch.cuda.synchronize()
    flushed_ms = statistics.median(a.elapsed_time(c) for a, c in fl)

    # ---- the same steps launched one call at a time ----
    eg = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K1)]
    for i in range(K1):
        flush()
        eg[i][0].record(stream)
        step()
        eg[i][1].record(stream)
    torch.cuda.synchronize()
    eager_ms = statistics.median(a.elapsed_time(c) for a, c in eg)

    # ---- per-call pass: each call timed alone, L2 flushed before it (roofline of the dominant call) ----
    K2 = min(K, 300)
    names = ["adaln_proj_fwd", "adaln_out_fwd", "adaln_out_bwd", "adaln_proj_bwd"]
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(4)]
          for _ in range(K2)]
    calls = [
        lambda: binding.adaln_proj_fwd(temb, W, b, emb=emb, u=u, stream=stream),
        lambda: binding.adaln_out_fwd(x, emb, out=out, mean=mean, rstd=rstd, stream=stream),
        lambda: binding.adaln_out_bwd(dy, x, emb, mean, rstd, dx=dx, d_emb=d_emb, workspace=ws_bwd, stream=stream),
        lambda: binding.adaln_proj_bwd(d_emb, temb, u, W, d_temb=d_temb, dW=dW, db=db, workspace=ws_proj,
                                       stream=stream),
    ]
    for i in range(K2):
        for j, c in enumerate(calls):
            flush()
            ev[i][j][0].record(stream)
            c()
            ev[i][j][1].record(stream)
    torch.cuda.synchronize()
    call_ms = {n: statistics.mean(ev[i][j][0].elapsed_time(ev[i][j][1]) for i in range(K2)) for j, n in enumerate(names)}

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

    e2e_sets = [dev_set(), dev_set()]

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
        d = e2e_sets[i % 2]
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
    peak, peak_src = hbm_peak()
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
        "ms_per_step_spread": {"min": min(passes) / K * 1e3, "max": max(passes) / K * 1e3, "passes": len(passes)},
        "ms_per_step_flushed": flushed_ms,
        "ms_per_step_eager": eager_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "compute": "fp32 arithmetic on bf16 tensors",
        "data": "synthetic (seeded; x, dy ~ N(0,1) with 81 outlier rows x50; W, b ~ N(0, 0.02^2))",
        "config": {"workload": "AdaLN norm_out fwd+bwd, B=2 S=4096 D=3072, 1% outlier rows",
                   "B": B, "S": S, "D": D, "parallelism": "replicas" if world > 1 else "single GPU",
                   "launch": ("eager: one C-ABI call at a time" if graphs is None else
                              "CUDA graphs of the step's four C-ABI calls (7 kernels, programmatic launch edges), "
                              "one per input set, captured once after the warm-up; K steps replayed back to back"),
                   "l2": ("inputs larger than L2: consecutive steps alternate between two copies of the inputs "
                          "(138 MB each, L2 129 MB), no flush; ms_per_step_flushed: the same step with a 512 MiB "
                          "write + 512 MiB read between steps, one event pair per step"),
                   "timing": f"median of {len(passes)} passes of K={K} steps (one event pair per pass), "
                             f"{wall:.2f} s timed in all"},
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
        "gpu_launches": KERNELS_PER_STEP * K,  # in the reported pass of K steps
        "clocks": {**clk, "bins": bins},
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


def run_chunking(args, rank, local):
    """The chunking workload: 4096 samples of S = 256 (D = 3072), forward and
    backward through the four calls, run as 1 x 4096, 2 x 2048, 16 x 256,
    64 x 64 and 4096 x 1 chunks, dW/db accumulated in fp32 over the chunks.  One
    JSON line per chunking on rank 0 (tokens/s over the whole workload, CUDA
    events around it, W warm-up runs first); every chunking's dW equals the
    first's bit for bit.  Inputs drawn on the device (seeded): x, dy, temb
    ~ N(0, 1), W, b ~ N(0, 0.02^2), all rounded to bf16."""
    if rank != 0:
        return
    import torch
    from invariant_dit_adaln_gb300 import binding, build

    torch.cuda.set_device(local)
    build.build()
    binding.load()
    n, S, D = 4096, 256, 3072
    N = 2 * D
    g = torch.Generator(device="cuda")
    g.manual_seed(WORKLOAD["seed"])
    x = torch.randn((n, S, D), generator=g, device="cuda").to(torch.bfloat16)
    dy = torch.randn((n, S, D), generator=g, device="cuda").to(torch.bfloat16)
    temb = torch.randn((n, D), generator=g, device="cuda").to(torch.bfloat16)
    W = (torch.randn((N, D), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    b = (torch.randn((N,), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    emb = torch.empty((n, N), dtype=torch.bfloat16, device="cuda")
    u = torch.empty((n, D), dtype=torch.bfloat16, device="cuda")
    out, dx = torch.empty_like(x), torch.empty_like(x)
    mean = torch.empty((n, S), device="cuda")
    rstd = torch.empty_like(mean)
    d_emb = torch.empty((n, N), device="cuda")
    d_temb = torch.empty_like(u)
    accW = torch.empty((N, D), device="cuda")
    accb = torch.empty((N,), device="cuda")
    ws1 = torch.empty(binding.adaln_out_bwd_workspace_bytes(n, S, D), dtype=torch.uint8, device="cuda")
    ws2 = torch.empty(binding.adaln_proj_bwd_workspace_bytes(n, D), dtype=torch.uint8, device="cuda")

    def run(chunk):
        for i in range(0, n, chunk):
            j = i + chunk
            binding.adaln_proj_fwd(temb[i:j], W, b, emb=emb[i:j], u=u[i:j])
            binding.adaln_out_fwd(x[i:j], emb[i:j], out=out[i:j], mean=mean[i:j], rstd=rstd[i:j])
            binding.adaln_out_bwd(dy[i:j], x[i:j], emb[i:j], mean[i:j], rstd[i:j], dx=dx[i:j], d_emb=d_emb[i:j],
                                  workspace=ws1)
            binding.adaln_proj_bwd(d_emb[i:j], temb[i:j], u[i:j], W, d_temb=d_temb[i:j], dW_acc=accW, db_acc=accb,
                                   accumulate=i > 0, workspace=ws2)

    ref = None
    for chunk in (4096, 2048, 256, 64, 1):
        for _ in range(max(1, min(args.warmup, 3))):
            run(chunk)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        run(chunk)
        e1.record()
        torch.cuda.synchronize()
        if binding.device_error() != 0:
            raise RuntimeError("device-side error in the chunking workload")
        sec = e0.elapsed_time(e1) / 1e3
        same = None
        if ref is None:
            ref = accW.clone()
        else:
            same = bool(torch.equal(accW.view(torch.int32), ref.view(torch.int32)))
        print(json.dumps({"workload": "chunking: 4096 samples of S=256, D=3072, fwd+bwd", "chunks": n // chunk,
                          "samples_per_chunk": chunk, "value": n * S / sec, "unit": "tokens/s", "ms": sec * 1e3,
                          "dW_bitwise_equal_to_1x4096": same, "data": "synthetic (seeded, drawn on the device)"}),
              flush=True)


def hbm_peak():
    """(GB/s, source): the measured copy bandwidth of MEASURED_PEAKS.json, else
    the machine's fallback figure."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
        if "hbm_gbs" in peaks:
            return float(peaks["hbm_gbs"]), "measured"
    except (OSError, ValueError):
        pass
    return 6800.0, "fallback"


def run_block(args, rank, local):
    """The block-level modulated norm with a gated residual
    (adaln_scale_residual_norm_fwd + _bwd with the residual output's later
    gradient) at B=2, S=4096, D=3072: K steps replayed from a CUDA graph, two
    input sets larger than L2 alternating, median of passes; one JSON line on
    rank 0 with tokens/s and the algorithmic HBM bytes of the pair (forward:
    x, residual read, r, out written, mean/rstd; backward: d_out, d_r, x, r
    read, d_x, d_residual written, stats), against the measured copy peak."""
    if rank != 0:
        return
    import torch
    from invariant_dit_adaln_gb300 import binding, build

    torch.cuda.set_device(local)
    build.build()
    binding.load()
    B, S, D = 2, 4096, 3072
    g = torch.Generator(device="cuda")
    g.manual_seed(WORKLOAD["seed"])

    def make():
        t = {k: torch.randn((B, S, D), generator=g, device="cuda").to(torch.bfloat16)
             for k in ("x", "residual", "dy", "dr")}
        t["gate"] = (torch.randn((B, D), generator=g, device="cuda") * 0.5).to(torch.bfloat16)
        t["emb"] = (torch.randn((B, 2 * D), generator=g, device="cuda") * 0.3).to(torch.bfloat16)
        for k in ("r", "out", "d_x", "d_res"):
            t[k] = torch.empty((B, S, D), dtype=torch.bfloat16, device="cuda")
        t["mean"], t["rstd"] = torch.empty((B, S), device="cuda"), torch.empty((B, S), device="cuda")
        t["d_emb"], t["d_gate"] = torch.empty((B, 2 * D), device="cuda"), torch.empty((B, D), device="cuda")
        t["ws"] = torch.empty(binding.adaln_scale_residual_norm_bwd_workspace_bytes(B, S, D), dtype=torch.uint8,
                              device="cuda")
        return t

    sets = [make(), make()]
    stream = torch.cuda.Stream()

    def step(t):
        binding.adaln_scale_residual_norm_fwd(t["x"], t["residual"], t["gate"], t["emb"], r=t["r"], out=t["out"],
                                              mean=t["mean"], rstd=t["rstd"], stream=stream)
        binding.adaln_scale_residual_norm_bwd(t["dy"], t["dr"], t["x"], t["r"], t["gate"], t["emb"], t["mean"],
                                              t["rstd"], d_x=t["d_x"], d_residual=t["d_res"], d_emb=t["d_emb"],
                                              d_gate=t["d_gate"], workspace=t["ws"], stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            for t in sets:
                step(t)
    torch.cuda.synchronize()
    graphs = []
    for t in sets:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            step(t)
        graphs.append(gr)
    torch.cuda.synchronize()
    K = min(args.steps, 2000)
    passes = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):  # replay() launches on the current stream: the events' stream
            e0.record(stream)
            for i in range(K):
                graphs[i % 2].replay()
            e1.record(stream)
        torch.cuda.synchronize()
        passes.append(e0.elapsed_time(e1) / K)
    if binding.device_error() != 0:
        raise RuntimeError("device-side error in the block-norm workload")
    ms = statistics.median(passes)
    alg = B * S * (4 * 2 * D + 8) + B * S * (6 * 2 * D + 8) + 4 * B * D * 2
    peak, peak_src = hbm_peak()
    print(json.dumps({"workload": "block-level modulated norm with a gated residual, fwd+bwd, B=2 S=4096 D=3072",
                      "value": B * S / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms,
                      "algorithmic_bytes_per_step": alg, "hbm_gbs": alg / (ms / 1e3) / 1e9,
                      "hbm_frac": alg / (ms / 1e3) / 1e9 / peak, "peak_gbs": peak, "peak_source": peak_src,
                      "kernels_per_step": 5, "steps_per_pass": K, "passes": len(passes),
                      "l2": "two input sets alternate (each: four 50.3 MB token inputs and four 50.3 MB token outputs, more than L2); no flush",
                      "data": "synthetic (seeded, drawn on the device)"}), flush=True)


def run_f32(args, rank, local):
    """The fp32 execution dtype: the whole step (adaln_f32_proj_fwd,
    adaln_f32_out_fwd, adaln_f32_out_bwd, adaln_f32_proj_bwd with dW, db) at
    B=2, S=4096, D=3072: K steps replayed from CUDA graphs over two input sets
    larger than L2, median of passes; one JSON line on rank 0 with tokens/s
    and the algorithmic HBM bytes against the measured copy peak."""
    if rank != 0:
        return
    import torch
    from invariant_dit_adaln_gb300 import binding, build

    torch.cuda.set_device(local)
    build.build()
    binding.load()
    B, S, D = 2, 4096, 3072
    N = 2 * D
    g = torch.Generator(device="cuda")
    g.manual_seed(WORKLOAD["seed"])
    W = torch.randn((N, D), generator=g, device="cuda") * 0.02
    bias = torch.randn((N,), generator=g, device="cuda") * 0.02

    def make():
        t = {"x": torch.randn((B, S, D), generator=g, device="cuda"),
             "dy": torch.randn((B, S, D), generator=g, device="cuda"),
             "temb": torch.randn((B, D), generator=g, device="cuda")}
        t["emb"], t["u"] = torch.empty((B, N), device="cuda"), torch.empty((B, D), device="cuda")
        t["out"], t["dx"] = torch.empty((B, S, D), device="cuda"), torch.empty((B, S, D), device="cuda")
        t["mean"], t["rstd"] = torch.empty((B, S), device="cuda"), torch.empty((B, S), device="cuda")
        t["d_emb"], t["d_temb"] = torch.empty((B, N), device="cuda"), torch.empty((B, D), device="cuda")
        t["dW"], t["db"] = torch.empty((N, D), device="cuda"), torch.empty((N,), device="cuda")
        t["ws1"] = torch.empty(binding.adaln_f32_out_bwd_workspace_bytes(B, S, D), dtype=torch.uint8, device="cuda")
        t["ws2"] = torch.empty(binding.adaln_f32_proj_bwd_workspace_bytes(B, D), dtype=torch.uint8, device="cuda")
        return t

    sets = [make(), make()]
    stream = torch.cuda.Stream()

    def step(t):
        binding.adaln_f32_proj_fwd(t["temb"], W, bias, emb=t["emb"], u=t["u"], stream=stream)
        binding.adaln_f32_out_fwd(t["x"], t["emb"], out=t["out"], mean=t["mean"], rstd=t["rstd"], stream=stream)
        binding.adaln_f32_out_bwd(t["dy"], t["x"], t["emb"], t["mean"], t["rstd"], dx=t["dx"], d_emb=t["d_emb"],
                                  workspace=t["ws1"], stream=stream)
        binding.adaln_f32_proj_bwd(t["d_emb"], t["temb"], t["u"], W, d_temb=t["d_temb"], dW_acc=t["dW"],
                                   db_acc=t["db"], workspace=t["ws2"], stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            for t in sets:
                step(t)
    torch.cuda.synchronize()
    graphs = []
    for t in sets:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            step(t)
        graphs.append(gr)
    torch.cuda.synchronize()
    K = min(args.steps, 1000)
    passes = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):  # replay() launches on the current stream: the events' stream
            e0.record(stream)
            for i in range(K):
                graphs[i % 2].replay()
            e1.record(stream)
        torch.cuda.synchronize()
        passes.append(e0.elapsed_time(e1) / K)
    if binding.device_error() != 0:
        raise RuntimeError("device-side error in the fp32 workload")
    ms = statistics.median(passes)
    tok, wb = B * S * D * 4, N * D * 4
    alg = (wb + N * 4 + 2 * B * D * 4 + B * N * 4          # projection forward
           + 2 * tok + B * S * 8 + B * N * 4                # LayerNorm forward
           + 3 * tok + B * S * 8 + 2 * B * N * 4            # LayerNorm backward
           + 2 * wb + N * 4 + B * N * 4 + 3 * B * D * 4)    # projection backward (dW, db written)
    peak, peak_src = hbm_peak()
    print(json.dumps({"workload": "fp32 execution dtype, fwd+bwd, B=2 S=4096 D=3072", "value": B * S / (ms / 1e3),
                      "unit": "tokens/s", "ms_per_step": ms, "algorithmic_bytes_per_step": alg,
                      "hbm_gbs": alg / (ms / 1e3) / 1e9, "hbm_frac": alg / (ms / 1e3) / 1e9 / peak, "peak_gbs": peak,
                      "peak_source": peak_src, "kernels_per_step": 7, "steps_per_pass": K, "passes": len(passes),
                      "l2": "two input sets alternate (x, dy 100.7 MB each per set, more than L2); no flush",
                      "dtype": "f32", "data": "synthetic (seeded, drawn on the device)"}), flush=True)


def run_proj_out(args, rank, local):
    """The forward with proj_out fused (adaln_out_fwd_proj) against the forward
    alone (adaln_out_fwd) at B=2, S=4096, D=3072, J=64: K calls of each
    replayed from CUDA graphs over two input sets larger than L2, median of
    passes; one JSON line on rank 0 with tokens/s of the fused call, the time
    y adds, and the fused call's algorithmic bytes (x read, out and y written,
    mean/rstd, Wp) against the measured copy peak."""
    if rank != 0:
        return
    import torch
    from invariant_dit_adaln_gb300 import binding, build

    torch.cuda.set_device(local)
    build.build()
    binding.load()
    B, S, D, J = 2, 4096, 3072, 64
    g = torch.Generator(device="cuda")
    g.manual_seed(WORKLOAD["seed"])
    Wp = (torch.randn((J, D), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    bp = (torch.randn((J,), generator=g, device="cuda") * 0.02).to(torch.bfloat16)

    def make():
        t = {"x": torch.randn((B, S, D), generator=g, device="cuda").to(torch.bfloat16),
             "emb": (torch.randn((B, 2 * D), generator=g, device="cuda") * 0.3).to(torch.bfloat16)}
        t["out"] = torch.empty((B, S, D), dtype=torch.bfloat16, device="cuda")
        t["y"] = torch.empty((B, S, J), dtype=torch.bfloat16, device="cuda")
        t["mean"], t["rstd"] = torch.empty((B, S), device="cuda"), torch.empty((B, S), device="cuda")
        return t

    sets = [make(), make()]
    stream = torch.cuda.Stream()

    def fused(t):
        binding.adaln_out_fwd_proj(t["x"], t["emb"], Wp, bp, out=t["out"], mean=t["mean"], rstd=t["rstd"], y=t["y"],
                                   stream=stream)

    def alone(t):
        binding.adaln_out_fwd(t["x"], t["emb"], out=t["out"], mean=t["mean"], rstd=t["rstd"], stream=stream)

    res = {}
    for name, fn in (("fused", fused), ("alone", alone)):
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                for t in sets:
                    fn(t)
        torch.cuda.synchronize()
        graphs = []
        for t in sets:
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                fn(t)
            graphs.append(gr)
        torch.cuda.synchronize()
        K = min(args.steps, 2000)
        passes = []
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                for i in range(K):
                    graphs[i % 2].replay()
                e1.record(stream)
            torch.cuda.synchronize()
            passes.append(e0.elapsed_time(e1) / K)
        res[name] = statistics.median(passes)
    if binding.device_error() != 0:
        raise RuntimeError("device-side error in the proj_out workload")
    ms = res["fused"]
    alg = B * S * (2 * D * 2 + 8 + J * 2) + J * D * 2 + B * 2 * D * 2
    peak, peak_src = hbm_peak()
    print(json.dumps({"workload": "forward with proj_out fused (D -> 64), B=2 S=4096 D=3072",
                      "value": B * S / (ms / 1e3), "unit": "tokens/s", "ms_per_call": ms,
                      "ms_forward_alone": res["alone"], "ms_added_by_proj_out": ms - res["alone"],
                      "algorithmic_bytes_per_call": alg, "hbm_gbs": alg / (ms / 1e3) / 1e9,
                      "hbm_frac": alg / (ms / 1e3) / 1e9 / peak, "peak_gbs": peak, "peak_source": peak_src,
                      "tflops_proj_out": 2.0 * B * S * D * J / ((ms - res["alone"]) / 1e3) / 1e12
                      if ms > res["alone"] else None,
                      "kernels_per_call": 2, "l2": "two input sets alternate (x 50.3 MB each); no flush",
                      "data": "synthetic (seeded, drawn on the device)"}), flush=True)


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
    ap.add_argument("--min-timed-s", type=float, default=1.5, help="repeat the K-step pass until this long is timed")
    ap.add_argument("--max-passes", type=int, default=2000)
    ap.add_argument("--proj-sweep", action="store_true",
                    help="instead of the step: time the projection calls alone for B = 1 .. 2048")
    ap.add_argument("--chunking", action="store_true",
                    help="instead of the step: the 4096-sample chunking workload in its five chunkings")
    ap.add_argument("--block", action="store_true",
                    help="instead of the step: the block-level modulated norm with a gated residual, fwd+bwd")
    ap.add_argument("--fp32", action="store_true", help="instead of the step: the fp32 execution dtype's step")
    ap.add_argument("--proj-out", action="store_true", help="instead of the step: the forward with proj_out fused")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_env()
    if args.proj_sweep:
        run_proj_sweep(args, rank, local)
        return
    if args.chunking:
        run_chunking(args, rank, local)
        return
    if args.block:
        run_block(args, rank, local)
        return
    if args.fp32:
        run_f32(args, rank, local)
        return
    if args.proj_out:
        run_proj_out(args, rank, local)
        return
    if args.impl == "reference":
        res = run_reference(args, world, rank)
    else:
        res = run_gpu(args, world, rank, local)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
