"""The fp32 execution dtype (adaln_f32_*) against the oracle, on the GPU.

Tolerances (tests/tolerance.py): fp32 outputs within 1e-5 relative of the
oracle's correctly rounded value, or within the floor of the fp32 arithmetic
that produces them (2^-16 of the sum of the absolute terms, as for the fp32
sums of the bf16 path).  Bit for bit where the operation fixes the fp32 order:
d_emb (the token trees, replayed from the GPU's own mean and rstd), dW and db
(the sequential fused multiply-add over samples, from the GPU's own u).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from invariant_dit_adaln_gb300 import binding
from gpu_util import dev_f32, host_f32, lib
from tolerance import F_OUT, F_RED, assert_bitwise, check_f32, floor_d_emb, floor_dx, floor_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    oracle.build()
    lib()
    yield
    assert binding.device_error() == 0


def _inputs(B, S, D, seed, outlier_frac=0.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, S, D)).astype(np.float32)
    dy = rng.standard_normal((B, S, D)).astype(np.float32)
    k = int(outlier_frac * B * S)
    if k:
        rows = rng.choice(B * S, k, replace=False)
        x.reshape(B * S, D)[rows] *= 50
        dy.reshape(B * S, D)[rows] *= 50
    return {"x": x, "dy": dy, "temb": rng.standard_normal((B, D)).astype(np.float32),
            "W": (rng.standard_normal((2 * D, D)) * 0.02).astype(np.float32),
            "b": (rng.standard_normal(2 * D) * 0.02).astype(np.float32)}


def _ulp32(a, b):
    ia = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    ib = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    ia = np.where(ia < 0, -(ia & 0x7FFFFFFF), ia)
    ib = np.where(ib < 0, -(ib & 0x7FFFFFFF), ib)
    return np.abs(ia - ib)


def _step(i, eps=1e-6):
    d = {k: dev_f32(v) for k, v in i.items()}
    emb, u = binding.adaln_f32_proj_fwd(d["temb"], d["W"], d["b"])
    out, mean, rstd = binding.adaln_f32_out_fwd(d["x"], emb, eps=eps)
    dx, d_emb = binding.adaln_f32_out_bwd(d["dy"], d["x"], emb, mean, rstd)
    d_temb, dW, db = binding.adaln_f32_proj_bwd(d_emb, d["temb"], u, d["W"])
    torch.cuda.synchronize()
    return {"emb": emb, "u": u, "out": out, "mean": mean, "rstd": rstd, "dx": dx, "d_emb": d_emb, "d_temb": d_temb,
            "dW": dW, "db": db}


def _check(i, g):
    h = {k: host_f32(v) for k, v in g.items()}
    B, S, D = i["x"].shape
    # projection: u within one ulp of the correctly rounded SiLU, emb staged on the GPU's u
    w_emb, w_u = oracle.f32_proj_fwd(i["temb"], i["W"], i["b"])
    dist = _ulp32(h["u"], w_u)
    assert dist.max() <= 1 and (dist == 0).mean() > 0.999, dist.max()
    e_emb, _ = oracle.f32_proj_fwd(i["temb"], i["W"], i["b"])
    fl_emb = F_OUT * (np.abs(h["u"].astype(np.float64)) @ np.abs(i["W"].astype(np.float64)).T
                      + np.abs(i["b"].astype(np.float64)))
    check_f32(h["emb"], e_emb, fl_emb, what="f32 emb")
    # LayerNorm + modulation, staged on the GPU's emb
    w_out, w_mean, w_rstd = oracle.f32_out_fwd(i["x"], h["emb"])
    xf = i["x"].astype(np.float64)
    onep = (np.float32(1) + h["emb"][:, :D]).astype(np.float64)
    check_f32(h["out"], w_out, floor_out(xf, onep, h["emb"][:, D:].astype(np.float64)), what="f32 out")
    check_f32(h["mean"], w_mean, F_RED * np.abs(xf).mean(-1), what="f32 mean")
    check_f32(h["rstd"], w_rstd, what="f32 rstd")
    # backward: dx within tolerance; d_emb bit for bit against the tree replay
    w_dx, w_demb = oracle.f32_out_bwd(i["dy"], i["x"], h["emb"])
    gf = i["dy"].astype(np.float64)
    check_f32(h["dx"], w_dx, floor_dx(xf, gf, onep), what="f32 dx")
    prod = oracle.f32_bwd_products(i["dy"], i["x"], h["mean"], h["rstd"])
    assert_bitwise(h["d_emb"], oracle.token_tree_f32(prod), "f32 d_emb vs fp32 tree replay")
    check_f32(h["d_emb"], w_demb, floor_d_emb(xf, gf), what="f32 d_emb vs fp64")
    # projection backward, staged on the GPU's d_emb and u
    w_dt, _, _ = oracle.f32_proj_bwd(h["d_emb"], i["temb"], i["W"], want_dW=False)
    t = i["temb"].astype(np.float64)
    s = 1.0 / (1.0 + np.exp(-t))
    fl_dt = F_OUT * (np.abs(h["d_emb"].astype(np.float64)) @ np.abs(i["W"].astype(np.float64))) * \
        np.abs(s * (1.0 + t * (1.0 - s)))
    check_f32(h["d_temb"], w_dt, fl_dt, what="f32 d_temb")
    sW, sb = oracle.f32_wgrad_seq(h["d_emb"], h["u"])
    assert_bitwise(h["dW"], sW, "f32 dW")
    assert_bitwise(h["db"], sb, "f32 db")


@pytest.mark.parametrize("B,S,D,seed,outl", [(2, 33, 3072, 0, 0.0), (1, 1, 3072, 1, 0.0), (2, 69, 3072, 2, 0.03),
                                             (3, 7, 256, 3, 0.0), (2, 40, 8, 4, 0.0), (5, 35, 520, 5, 0.0),
                                             (1, 33, 4096, 6, 0.0)])
def test_f32_step(B, S, D, seed, outl):
    i = _inputs(B, S, D, seed, outl)
    _check(i, _step(i))


def test_f32_step_full_size():
    """B=2, S=4096, D=3072 with 1 % outlier rows: every element."""
    i = _inputs(2, 4096, 3072, 7, 0.01)
    _check(i, _step(i))


def test_f32_rows_do_not_depend_on_the_batch():
    """Every per-sample output of sample b has the same bytes in a batch of 3
    and alone; dW, db of the batch equal the samples accumulated one by one."""
    i = _inputs(3, 45, 3072, 8)
    full = _step(i)
    D = 3072
    accW = torch.empty((2 * D, D), device="cuda")
    accb = torch.empty((2 * D,), device="cuda")
    for b in range(3):
        one = _step({k: (v[b:b + 1] if k in ("x", "dy", "temb") else v) for k, v in i.items()})
        for k in ("emb", "u", "out", "mean", "rstd", "dx", "d_emb", "d_temb"):
            assert torch.equal(full[k][b:b + 1].view(torch.int32), one[k].view(torch.int32)), (b, k)
        binding.adaln_f32_proj_bwd(full["d_emb"][b:b + 1], dev_f32(i["temb"][b:b + 1]), full["u"][b:b + 1],
                                   dev_f32(i["W"]), dW_acc=accW, db_acc=accb, accumulate=b > 0)
    torch.cuda.synchronize()
    assert torch.equal(accW.view(torch.int32), full["dW"].view(torch.int32))
    assert torch.equal(accb.view(torch.int32), full["db"].view(torch.int32))
