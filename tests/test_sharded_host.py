"""Host logic of the sample-sharded step (invariant_dit_adaln_gb300.sharded) on
the CPU with two gloo ranks.

The compute is the oracle (a test double of the library's calls), so these
tests check the plan and the data movement: every output row of the weight
gradient is owned by exactly one rank, in ascending order; the gathered d_emb
and u hold all samples in ascending order; and the row blocks of dW and db,
concatenated in rank order, are bit for bit the gradient of the whole batch in
the sequential order.  The GPU side (adaln_proj_wgrad_rows giving the rows of
adaln_proj_bwd's gradient) is tested in test_gpu_parity.py.
"""

from __future__ import annotations

import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from invariant_dit_adaln_gb300 import sharded, synth

B, S, D = 5, 33, 16


def test_plan_owns_every_row_and_sample_once():
    for world in (1, 2, 3, 4, 7):
        for b in (1, 5, 8, 13):
            plans = [sharded.ShardPlan.make(b, D, world, r) for r in range(world)]
            rows = [n for p in plans for n in range(*p.rows)]
            assert rows == list(range(2 * D))
            samples = [i for p in plans for i in range(*p.samples)]
            assert samples == list(range(b))
            assert sum(plans[0].sample_counts) == b


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16))


class OracleOps:
    """The library's calls on the CPU oracle; bf16 tensors as int16 bit tensors."""

    def __init__(self, temb_all):
        import oracle
        oracle.build()
        self.o = oracle
        self.temb_all = temb_all

    def forward(self, x, temb, W, bias):
        emb = self.o.proj_fwd(_bits(temb), _bits(W), _bits(bias))
        u = self.o.silu_bf16(_bits(temb))
        out, mean, rstd = self.o.out_fwd(_bits(x), emb)
        return _t(emb), _t(u), _t(out), torch.from_numpy(mean), torch.from_numpy(rstd)

    def backward(self, dy, x, emb, mean, rstd, temb, u, W):
        dx, d_emb = self.o.out_bwd(_bits(dy), _bits(x), _bits(emb))
        d_temb, _, _ = self.o.proj_bwd(d_emb, _bits(temb), _bits(W), want_dW=False)
        return _t(dx), torch.from_numpy(d_emb), _t(d_temb)

    def wgrad_rows(self, d_emb_all, u_all, n0, n1):
        dW, db = self.o.wgrad_seq_f32_rows(d_emb_all.numpy(), self.temb_all, np.arange(n0, n1, dtype=np.int32))
        return _t(synth.bf16_bits_from_f32(dW)), _t(synth.bf16_bits_from_f32(db))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    inp = synth.make_inputs(B, S, D, 7, outlier_frac=0.05)
    plan = sharded.ShardPlan.make(B, D, world, rank)
    s0, s1 = plan.samples
    r = sharded.sharded_step(_t(inp["x"][s0:s1]), _t(inp["dy"][s0:s1]), _t(inp["temb"][s0:s1]), _t(inp["W"]),
                             _t(inp["b"]), plan, dist, ops=OracleOps(inp["temb"]))
    q.put((rank, plan.rows, r["d_emb_all"].numpy(), _bits(r["u_all"]), _bits(r["dW_rows"]), _bits(r["db_rows"]),
           r["d_emb"].numpy()))
    dist.barrier()
    dist.destroy_process_group()


def test_sharded_step_with_two_gloo_ranks():
    import oracle
    oracle.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = []
    for _ in range(2):
        try:
            got.append(q.get(timeout=120))
        except Exception:
            break
    for p in procs:
        p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got.sort(key=lambda g: g[0])
    inp = synth.make_inputs(B, S, D, 7, outlier_frac=0.05)
    _, d_emb_full = oracle.out_bwd(inp["dy"], inp["x"], oracle.proj_fwd(inp["temb"], inp["W"], inp["b"]))
    for rank, rows, d_emb_all, u_all, _, _, d_emb_local in got:
        # the gathered tensors hold every sample in ascending order
        assert np.array_equal(d_emb_all.view(np.uint32), d_emb_full.view(np.uint32)), rank
        assert np.array_equal(u_all, oracle.silu_bf16(inp["temb"])), rank
    # each rank's own samples are its block of the batch
    assert np.array_equal(np.concatenate([g[6] for g in got]).view(np.uint32), d_emb_full.view(np.uint32))
    # the row blocks, in rank order, are the whole batch's gradient bit for bit
    assert [g[1] for g in got] == [(0, D), (D, 2 * D)]
    dW_full, db_full = oracle.wgrad_seq_f32(d_emb_full, inp["temb"])
    assert np.array_equal(np.concatenate([g[4] for g in got]), synth.bf16_bits_from_f32(dW_full))
    assert np.array_equal(np.concatenate([g[5] for g in got]), synth.bf16_bits_from_f32(db_full))
