"""The block-level modulated norm with a gated residual
(adaln_scale_residual_norm_fwd / _bwd) against the oracle, on the GPU.

Staged like the other parity tests: the backward's tail is checked given the
GPU's own LayerNorm input gradient (the dx of adaln_out_bwd at r, the same
kernels), so that one rounding difference upstream cannot cascade.  Bit for
bit where the operation fixes every rounding: r (two eager bf16 roundings),
d_residual, d_x, the tree replay of d_gate and of d_emb.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from invariant_dit_adaln_gb300 import binding, synth
from gpu_util import dev_bf16, host_bf16, host_f32, lib
from tolerance import (F_RED, F_TREE_ABS, F_TREE_REL, assert_bitwise, bf16_to_f64, check_bf16, check_f32,
                       floor_d_emb, floor_dx, floor_out)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    oracle.build()
    lib()
    yield
    assert binding.device_error() == 0


def _onep_shift(emb_bits, D):
    scale = bf16_to_f64(emb_bits[:, :D]).astype(np.float32)
    onep = bf16_to_f64(synth.bf16_bits_from_f32(np.float32(1) + scale))
    return onep, bf16_to_f64(emb_bits[:, D:])


def _dev(i):
    return {k: dev_bf16(v) for k, v in i.items() if k != "outlier_rows"}


def _gate_floor(prod):
    p = prod.astype(np.float64)
    return F_TREE_REL * np.abs(p.sum(axis=1)) + F_TREE_ABS * np.abs(p).sum(axis=1)


def _check_case(i, with_dr=True):
    B, S, D = i["x"].shape
    d = _dev(i)
    r, out, mean, rstd = binding.adaln_scale_residual_norm_fwd(d["x"], d["residual"], d["gate"], d["emb"])
    torch.cuda.synchronize()
    # forward: r bit for bit; out, mean, rstd as the norm_out forward of r
    w_r, w_out, w_mean, w_rstd = oracle.res_fwd(i["x"], i["residual"], i["gate"], i["emb"])
    assert_bitwise(host_bf16(r), w_r, "r")
    rf = bf16_to_f64(w_r)
    onep, shift = _onep_shift(i["emb"], D)
    st = check_bf16(host_bf16(out), w_out, floor_out(rf, onep, shift), what="block norm out")
    assert st["exact"] >= 0.95 * st["n"], st
    check_f32(host_f32(mean), w_mean, F_RED * np.abs(rf).mean(-1), what="block norm mean")
    check_f32(host_f32(rstd), w_rstd, what="block norm rstd")
    # backward
    d_r = d["dr"] if with_dr else None
    d_x, d_res, d_emb, d_gate = binding.adaln_scale_residual_norm_bwd(d["dy"], d_r, d["x"], r, d["gate"], d["emb"],
                                                                      mean, rstd)
    dr_ln, d_emb2 = binding.adaln_out_bwd(d["dy"], r, d["emb"], mean, rstd)
    torch.cuda.synchronize()
    assert_bitwise(host_f32(d_emb), host_f32(d_emb2), "d_emb = the norm_out backward's at r")
    prod = oracle.bwd_products_f32(i["dy"], w_r, host_f32(mean), host_f32(rstd))
    assert_bitwise(host_f32(d_emb), oracle.token_tree_f32(prod), "d_emb vs fp32 tree replay")
    gf = bf16_to_f64(i["dy"])
    w_dx, w_demb = oracle.out_bwd(i["dy"], w_r, i["emb"])
    check_bf16(host_bf16(dr_ln), w_dx, floor_dx(rf, gf, onep), what="dr_ln")
    check_f32(host_f32(d_emb), w_demb, floor_d_emb(rf, gf), what="block norm d_emb")
    # the tail, given the GPU's dr_ln: bit for bit
    t_dx, t_dres, t_dgate = oracle.res_bwd_tail(host_bf16(dr_ln), i["dr"] if with_dr else None, i["x"], i["gate"])
    assert_bitwise(host_bf16(d_res), t_dres, "d_residual")
    assert_bitwise(host_bf16(d_x), t_dx, "d_x")
    gprod = oracle.res_gate_products_f32(host_bf16(d_res), i["x"])
    assert_bitwise(host_f32(d_gate), oracle.token_tree_f32(gprod), "d_gate vs fp32 tree replay")
    check_f32(host_f32(d_gate), t_dgate, _gate_floor(gprod), what="d_gate vs fp64")
    return {"r": r, "out": out, "mean": mean, "rstd": rstd, "d_x": d_x, "d_res": d_res, "d_emb": d_emb,
            "d_gate": d_gate}


@pytest.mark.parametrize("B,S,D,seed,outl", [(2, 33, 3072, 0, 0.0), (1, 1, 3072, 1, 0.0), (2, 69, 3072, 2, 0.03),
                                             (3, 7, 256, 3, 0.0), (2, 40, 8, 4, 0.0), (1, 35, 4104, 5, 0.0),
                                             (2, 1100, 64, 6, 0.0), (2, 50, 2048, 10, 0.0), (1, 40, 4096, 11, 0.02),
                                             (2, 600, 3072, 12, 0.0)])
def test_scale_residual_norm(B, S, D, seed, outl):
    """The forward forms r inside the LayerNorm kernel up to D = 4096 (16 warps
    with one or two stages, or 8 warps at D = 4096; at S = 600 some warps of a
    CTA have no row) and with a separate gated-add kernel beyond (D = 4104)."""
    _check_case(synth.make_block_inputs(B, S, D, seed, outlier_frac=outl))


def test_scale_residual_norm_without_later_use():
    _check_case(synth.make_block_inputs(2, 37, 3072, 7), with_dr=False)


def test_scale_residual_norm_full_size():
    """B=2, S=4096, D=3072 with 1 % outlier rows: every element of r, d_x,
    d_residual, d_emb and d_gate bit for bit, out and dr_ln within tolerance."""
    _check_case(synth.make_block_inputs(2, 4096, 3072, 8, outlier_frac=0.01))


def test_scale_residual_norm_rows_do_not_depend_on_the_batch():
    """Every output of sample b has the same bytes in a batch of 3 and alone."""
    i = synth.make_block_inputs(3, 45, 3072, 9)
    d = _dev(i)

    def run(sl):
        r, out, mean, rstd = binding.adaln_scale_residual_norm_fwd(d["x"][sl], d["residual"][sl], d["gate"][sl],
                                                                   d["emb"][sl])
        d_x, d_res, d_emb, d_gate = binding.adaln_scale_residual_norm_bwd(d["dy"][sl], d["dr"][sl], d["x"][sl], r,
                                                                          d["gate"][sl], d["emb"][sl], mean, rstd)
        return [r, out, mean, rstd, d_x, d_res, d_emb, d_gate]

    full = run(slice(0, 3))
    for b in range(3):
        one = run(slice(b, b + 1))
        for k, (a, c) in enumerate(zip(full, one)):
            assert torch.equal(a[b:b + 1].contiguous().view(torch.uint8), c.view(torch.uint8)), (b, k)


def test_scale_residual_norm_empty_sequence():
    D = 256
    z = torch.zeros((2, 0, D), dtype=torch.bfloat16, device="cuda")
    gate = dev_bf16(np.zeros((2, D), np.uint16))
    emb = dev_bf16(np.zeros((2, 2 * D), np.uint16))
    r, out, mean, rstd = binding.adaln_scale_residual_norm_fwd(z, z, gate, emb)
    assert r.numel() == 0 and out.numel() == 0
    d_emb = torch.full((2, 2 * D), float("nan"), device="cuda")
    d_gate = torch.full((2, D), float("nan"), device="cuda")
    _, _, d_emb, d_gate = binding.adaln_scale_residual_norm_bwd(z, None, z, z, gate, emb, mean, rstd, d_emb=d_emb,
                                                                d_gate=d_gate)
    torch.cuda.synchronize()
    assert torch.all(d_emb == 0) and torch.all(d_gate == 0)
