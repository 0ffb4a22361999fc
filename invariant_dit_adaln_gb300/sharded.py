"""Sample-sharded data-parallel step of the AdaLN norm_out operator.

Each rank owns a contiguous block of the samples (ascending by rank) and runs
the LayerNorm forward and backward, the token trees and the projections for
them with the full W; rows never interact, and the token tree is per sample, so
nothing is exchanged for these.  The weight gradient sums over every sample, so
the ranks all-gather d_emb and u (in ascending sample order) and each rank
computes dW and db for its own block of output rows, over all samples in the
same ascending sequential order as one GPU.  No partial sums are reduced
across GPUs (miles_diffusion PR 108, second rendering, "Patches": bitwise
parity holds when nothing is reduced across ranks), so the concatenated row
blocks are the bytes of the one-GPU gradient.

The compute goes through an `ops` object; the default calls the CUDA library
(invariant_dit_adaln_gb300.binding).  This module only plans the shards and
moves tensors with torch.distributed.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch


def block(total: int, parts: int, i: int) -> tuple[int, int]:
    """[begin, end) of part i when `total` items are cut into `parts`
    contiguous blocks in ascending order (sizes differ by at most one)."""
    return total * i // parts, total * (i + 1) // parts


@dataclass(frozen=True)
class ShardPlan:
    """Which samples and which output rows of the weight gradient a rank owns."""
    samples: tuple[int, int]
    rows: tuple[int, int]
    sample_counts: tuple[int, ...]

    @staticmethod
    def make(B: int, D: int, world: int, rank: int) -> "ShardPlan":
        counts = tuple(block(B, world, r)[1] - block(B, world, r)[0] for r in range(world))
        return ShardPlan(samples=block(B, world, rank), rows=block(2 * D, world, rank), sample_counts=counts)


def gather_samples(local: torch.Tensor, counts, dist) -> torch.Tensor:
    """All ranks' blocks of samples (dimension 0), concatenated in rank order,
    which is the ascending global sample order.  Blocks may differ in size by
    one: each is padded to the largest before the all-gather, then trimmed."""
    world = len(counts)
    if world == 1:
        return local
    m = max(counts)
    # moved as raw bytes, so that any dtype goes through any backend
    row_bytes = local.element_size()
    for n in local.shape[1:]:
        row_bytes *= n
    raw = local.contiguous().view(torch.uint8).reshape(local.shape[0], row_bytes)
    pad = torch.zeros((m, row_bytes), dtype=torch.uint8, device=local.device)
    pad[: raw.shape[0]] = raw
    parts = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(parts, pad)
    out = torch.cat([p[:c] for p, c in zip(parts, counts)], dim=0)
    return out.view(local.dtype).reshape((sum(counts),) + tuple(local.shape[1:]))


class LibraryOps:
    """The compute of the sharded step, through the CUDA library."""

    def __init__(self):
        from . import binding
        self.b = binding

    def forward(self, x, temb, W, bias):
        emb, u = self.b.adaln_proj_fwd(temb, W, bias)
        out, mean, rstd = self.b.adaln_out_fwd(x, emb)
        return emb, u, out, mean, rstd

    def backward(self, dy, x, emb, mean, rstd, temb, u, W):
        dx, d_emb = self.b.adaln_out_bwd(dy, x, emb, mean, rstd)
        d_temb, _, _, _, _ = self.b.adaln_proj_bwd(d_emb, temb, u, W)
        return dx, d_emb, d_temb

    def wgrad_rows(self, d_emb_all, u_all, n0, n1):
        D = u_all.shape[1]
        dW = torch.empty((n1 - n0, D), dtype=torch.bfloat16, device=u_all.device)
        db = torch.empty((n1 - n0,), dtype=torch.bfloat16, device=u_all.device)
        _, _, dW, db = self.b.adaln_proj_wgrad_rows(d_emb_all, u_all, n0, n1, dW=dW, db=db)
        return dW, db


def sharded_step(x, dy, temb, W, bias, plan: ShardPlan, dist, ops=None):
    """One forward + backward of this rank's samples (x, dy, temb are its
    block).  Returns the per-sample results of its samples, the gathered d_emb
    and u of all samples, and its rows [n0, n1) of dW and db."""
    ops = ops or LibraryOps()
    emb, u, out, mean, rstd = ops.forward(x, temb, W, bias)
    dx, d_emb, d_temb = ops.backward(dy, x, emb, mean, rstd, temb, u, W)
    d_emb_all = gather_samples(d_emb, plan.sample_counts, dist)
    u_all = gather_samples(u, plan.sample_counts, dist)
    n0, n1 = plan.rows
    dW_rows, db_rows = ops.wgrad_rows(d_emb_all, u_all, n0, n1)
    return {"emb": emb, "u": u, "out": out, "mean": mean, "rstd": rstd, "dx": dx, "d_emb": d_emb, "d_temb": d_temb,
            "d_emb_all": d_emb_all, "u_all": u_all, "dW_rows": dW_rows, "db_rows": db_rows}
