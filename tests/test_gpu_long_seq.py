"""Parity of the whole fwd+bwd step at the long sequences of the pages' weight-
gradient failure case (S = 6032 and 6889, B = 2, D = 3072, 1 % outlier rows).

Both lengths end in a ragged tile (16 and 9 tokens) and fold through three
tree levels.  d_emb is compared bit for bit against the fp32 replay of the
token tree and within tolerance against the fp64 sums; dW and db bit for bit
against the sequential fp32 replay over the samples; d_temb and emb in full;
out, mean, rstd and dx on sampled rows (tile edges, the ragged last tile,
outlier rows and seeded random rows), each computed by the oracle row by row."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from invariant_dit_adaln_gb300 import binding, synth
from gpu_util import host_bf16, host_f32, lib, run_step, to_device
from tolerance import (F_RED, assert_bitwise, bf16_to_f64, check_bf16, check_f32, floor_d_emb, floor_d_temb, floor_dx,
                       floor_out)

pytestmark = pytest.mark.gpu

B, D = 2, 3072


@pytest.fixture(scope="module", params=[6032, 6889])
def run(request):
    S = request.param
    oracle.build()
    lib()
    inp = synth.make_inputs(B, S, D, 1, outlier_frac=0.01)
    r = run_step(to_device(inp))
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    return S, inp, {k: (host_bf16(v) if v.dtype == torch.bfloat16 else host_f32(v)) for k, v in r.items()}


def _sample_rows(S, inp):
    rng = np.random.default_rng(S)
    last = (S - 1) // 32 * 32  # first token of the ragged last tile
    rows = {0, 31, 32, 1023, 1024, last - 1, last, S - 2, S - 1}
    picked = {(int(f) // S, int(f) % S) for f in inp["outlier_rows"][:6]}
    for b in range(B):
        picked |= {(b, s) for s in rows}
        picked |= {(b, int(s)) for s in rng.integers(0, S, 6)}
    return sorted(picked)


def test_emb_and_u(run):
    S, inp, g = run
    check_bf16(g["emb"], oracle.proj_fwd(inp["temb"], inp["W"], inp["b"]), what="emb")
    assert_bitwise(g["u"], oracle.silu_bf16(inp["temb"]), "u")


def test_out_and_dx_sampled_rows(run):
    S, inp, g = run
    emb = g["emb"]
    onep_all = bf16_to_f64(synth.bf16_bits_from_f32(np.float32(1) + bf16_to_f64(emb[:, :D]).astype(np.float32)))
    for b, s in _sample_rows(S, inp):
        x = inp["x"][b:b + 1, s:s + 1]
        dy = inp["dy"][b:b + 1, s:s + 1]
        e = emb[b:b + 1]
        onep, shift = onep_all[b:b + 1], bf16_to_f64(e[:, D:])
        xf = bf16_to_f64(x)
        w_out, w_mean, w_rstd = oracle.out_fwd(x, e)
        check_bf16(g["out"][b:b + 1, s:s + 1], w_out, floor_out(xf, onep, shift), what=f"out row ({b},{s})")
        check_f32(g["mean"][b:b + 1, s:s + 1], w_mean, F_RED * np.abs(xf).mean(-1), what="mean")
        check_f32(g["rstd"][b:b + 1, s:s + 1], w_rstd, what="rstd")
        w_dx, _ = oracle.out_bwd(dy, x, e)
        check_bf16(g["dx"][b:b + 1, s:s + 1], w_dx, floor_dx(xf, bf16_to_f64(dy), onep), what=f"dx row ({b},{s})")


def test_d_emb(run):
    S, inp, g = run
    prod = oracle.bwd_products_f32(inp["dy"], inp["x"], g["mean"], g["rstd"])
    assert_bitwise(g["d_emb"], oracle.token_tree_f32(prod), f"d_emb vs fp32 tree replay, S={S}")
    _, w_demb = oracle.out_bwd(inp["dy"], inp["x"], g["emb"])
    check_f32(g["d_emb"], w_demb, floor_d_emb(bf16_to_f64(inp["x"]), bf16_to_f64(inp["dy"])), what="d_emb vs fp64")


def test_weight_gradients(run):
    S, inp, g = run
    d_emb = g["d_emb"]
    s_dW, s_db = oracle.wgrad_seq_f32(d_emb, inp["temb"])
    assert_bitwise(g["dW"], synth.bf16_bits_from_f32(s_dW), f"dW, S={S}")
    assert_bitwise(g["db"], synth.bf16_bits_from_f32(s_db), f"db, S={S}")
    w_dt, _, _ = oracle.proj_bwd(d_emb, inp["temb"], inp["W"], want_dW=False)
    fl = floor_d_temb(bf16_to_f64(synth.bf16_bits_from_f32(d_emb)), bf16_to_f64(inp["W"]),
                      oracle.dsilu_f64(bf16_to_f64(inp["temb"])))
    check_bf16(g["d_temb"], w_dt, fl, what="d_temb")
