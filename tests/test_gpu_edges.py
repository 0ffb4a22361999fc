"""Edge cases of the GPU path against the oracle: the longest sequence the ABI
accepts (the token tree at its deepest), empty forward calls, and the
projections at the largest D."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from invariant_dit_adaln_gb300 import binding, synth
from gpu_util import dev_bf16, dev_f32, host_bf16, host_f32, lib
from tolerance import assert_bitwise, bf16_to_f64, check_bf16, check_f32, floor_d_emb, floor_d_temb, floor_dx, floor_emb, floor_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    oracle.build()
    lib()
    yield
    assert binding.device_error() == 0


def _onep_shift(emb, D):
    onep = bf16_to_f64(synth.bf16_bits_from_f32(np.float32(1) + bf16_to_f64(emb[:, :D]).astype(np.float32)))
    return onep, bf16_to_f64(emb[:, D:])


def test_longest_sequence():
    """S = 262144 (32^3 * 8, the limit): 8192 tiles, four tree levels."""
    B, S, D = 1, 262144, 8
    inp = synth.make_inputs(B, S, D, 3, outlier_frac=0.01)
    emb = synth.normal_bf16(synth.stream_key(3, "aux"), B * 2 * D, std=0.3).reshape(B, 2 * D)
    x, dy = dev_bf16(inp["x"]), dev_bf16(inp["dy"])
    out, mean, rstd = binding.adaln_out_fwd(x, dev_bf16(emb))
    dx, d_emb = binding.adaln_out_bwd(dy, x, dev_bf16(emb), mean, rstd)
    torch.cuda.synchronize()
    xf, gf = bf16_to_f64(inp["x"]), bf16_to_f64(inp["dy"])
    onep, shift = _onep_shift(emb, D)
    w_out, _, _ = oracle.out_fwd(inp["x"], emb)
    check_bf16(host_bf16(out), w_out, floor_out(xf, onep, shift), what="out")
    w_dx, w_demb = oracle.out_bwd(inp["dy"], inp["x"], emb)
    check_bf16(host_bf16(dx), w_dx, floor_dx(xf, gf, onep), what="dx")
    prod = oracle.bwd_products_f32(inp["dy"], inp["x"], host_f32(mean), host_f32(rstd))
    assert_bitwise(host_f32(d_emb), oracle.token_tree_f32(prod), "d_emb vs fp32 tree replay, S=262144")
    check_f32(host_f32(d_emb), w_demb, floor_d_emb(xf, gf), what="d_emb vs fp64")


@pytest.mark.parametrize("B,S", [(0, 5), (3, 0), (0, 0)])
def test_empty_forward_writes_nothing(B, S):
    D = 64
    x = torch.zeros((B, S, D), dtype=torch.bfloat16, device="cuda")
    emb = torch.zeros((B, 2 * D), dtype=torch.bfloat16, device="cuda")
    out, mean, rstd = binding.adaln_out_fwd(x, emb)
    assert out.numel() == 0 and mean.numel() == 0 and rstd.numel() == 0
    temb = torch.zeros((0, D), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((2 * D, D), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros((2 * D,), dtype=torch.bfloat16, device="cuda")
    e, u = binding.adaln_proj_fwd(temb, W, b)
    assert e.numel() == 0 and u.numel() == 0


def test_projections_at_the_largest_D():
    B, D = 2, 8192
    inp = synth.make_inputs(B, 1, D, 8)
    temb, W, b = dev_bf16(inp["temb"]), dev_bf16(inp["W"]), dev_bf16(inp["b"])
    emb, u = binding.adaln_proj_fwd(temb, W, b)
    torch.cuda.synchronize()
    u_ref = oracle.silu_bf16(inp["temb"])
    assert_bitwise(host_bf16(u), u_ref, "u")
    fl = floor_emb(bf16_to_f64(u_ref), bf16_to_f64(inp["W"]), bf16_to_f64(inp["b"]))
    st = check_bf16(host_bf16(emb), oracle.proj_fwd(inp["temb"], inp["W"], inp["b"]), fl, what="emb")
    assert st["exact"] >= 0.99 * st["n"], st
    d_emb = synth.normal(synth.stream_key(8, "aux"), B * 2 * D).astype(np.float32).reshape(B, 2 * D)
    N = 2 * D
    dW = torch.empty((N, D), dtype=torch.bfloat16, device="cuda")
    db = torch.empty((N,), dtype=torch.bfloat16, device="cuda")
    d_temb, _, _, dW, db = binding.adaln_proj_bwd(dev_f32(d_emb), temb, u, W, dW=dW, db=db)
    torch.cuda.synchronize()
    s_dW, s_db = oracle.wgrad_seq_f32(d_emb, inp["temb"])
    assert_bitwise(host_bf16(dW), synth.bf16_bits_from_f32(s_dW), "dW")
    assert_bitwise(host_bf16(db), synth.bf16_bits_from_f32(s_db), "db")
    w_dt, _, _ = oracle.proj_bwd(d_emb, inp["temb"], inp["W"], want_dW=False)
    fl = floor_d_temb(bf16_to_f64(synth.bf16_bits_from_f32(d_emb)), bf16_to_f64(inp["W"]),
                      oracle.dsilu_f64(bf16_to_f64(inp["temb"])))
    st = check_bf16(host_bf16(d_temb), w_dt, fl, what="d_temb")
    assert st["exact"] >= 0.95 * st["n"], st
