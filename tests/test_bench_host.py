"""Host logic of bench.py on the CPU: byte accounting, whole-job throughput,
and the max-over-ranks timing across two gloo ranks (the replica layout: each
rank runs its own copy of the workload, no data-path collective)."""

from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def test_step_bytes_of_the_workload():
    B, S, D = bench.WORKLOAD["B"], bench.WORKLOAD["S"], bench.WORKLOAD["D"]
    cb = bench.call_bytes(B, S, D)
    rows, N = B * S, 2 * D
    # LayerNorm backward: read dy, x, emb, mean, rstd; write dx and d_emb
    assert cb["adaln_out_bwd"] == 2 * rows * D * 2 + B * N * 2 + 2 * rows * 4 + rows * D * 2 + B * N * 4
    assert bench.step_bytes(B, S, D) == sum(cb.values()) == 365293568


def test_throughput_is_whole_job():
    assert bench.throughput(8192 * 10, 1, 2.0) == 8192 * 10 / 2.0
    assert bench.throughput(8192 * 10, 4, 2.0) == 4 * 8192 * 10 / 2.0


def test_reference_arm_runs_on_rank_zero_only():
    class A:
        steps, warmup, ref_budget = 1, 3, 1.0
    assert bench.run_reference(A(), 2, 1) is None


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    w, r, _ = bench.dist_env()
    d = bench.init_dist(w, "gloo")
    bench.barrier(d)
    my_time = 1.0 + rank  # rank 1 is the slower one
    t_max = bench.max_over_ranks(my_time, d)
    q.put((r, t_max, bench.throughput(100, w, t_max)))
    bench.barrier(d)
    d.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] == 2.0 for g in got)           # every rank sees the max
    assert all(g[2] == 100 * 2 / 2.0 for g in got)  # units of all ranks over the max time
