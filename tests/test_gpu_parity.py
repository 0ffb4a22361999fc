"""Parity of every C-ABI entry point with the CPU oracle, element by element,
on the same seeded inputs.

Tolerances (tests/tolerance.py): bf16 outputs within one bf16 ulp of the
oracle's correctly rounded value, or within the error-bound floor of the fp32
arithmetic that produces them; fp32 outputs within 1e-5 relative or the floor.
Staged checks feed both sides the same intermediate (the GPU's emb, mean,
rstd, d_emb), so one rounding difference upstream cannot cascade.  Where the
operator fixes the fp32 order (the token tree, the weight gradient, the SiLU
rounding), the result must be bit-identical to the oracle's replay of it.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from invariant_dit_adaln_gb300 import binding, synth
from gpu_util import dev_bf16, dev_f32, host_bf16, host_f32, lib, to_device
from tolerance import (assert_bitwise, bf16_to_f64, check_bf16, check_f32, floor_d_emb, floor_d_temb, floor_dx,
                       floor_emb, floor_out, F_RED)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    oracle.build()
    lib()
    yield
    assert binding.device_error() == 0


def onep_shift(emb_bits, D):
    scale = bf16_to_f64(emb_bits[:, :D]).astype(np.float32)
    onep = bf16_to_f64(synth.bf16_bits_from_f32(np.float32(1) + scale))
    return onep, bf16_to_f64(emb_bits[:, D:])


# ---------------------------------------------------------------------------
# projection forward
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("B,D,seed", [(2, 3072, 0), (1, 3072, 1), (3, 3072, 2), (5, 512, 3), (9, 1024, 4),
                                      (2, 8, 5), (2, 4104, 6)])
def test_proj_fwd(B, D, seed):
    inp = synth.make_inputs(B, 1, D, seed)
    emb, u = binding.adaln_proj_fwd(dev_bf16(inp["temb"]), dev_bf16(inp["W"]), dev_bf16(inp["b"]))
    torch.cuda.synchronize()
    u_ref = oracle.silu_bf16(inp["temb"])
    assert_bitwise(host_bf16(u), u_ref, "u = bf16(silu(temb))")
    want = oracle.proj_fwd(inp["temb"], inp["W"], inp["b"])
    fl = floor_emb(bf16_to_f64(u_ref), bf16_to_f64(inp["W"]), bf16_to_f64(inp["b"]))
    st = check_bf16(host_bf16(emb), want, fl, what="emb")
    assert st["exact"] >= 0.99 * st["n"], st


def test_silu_every_bf16_input():
    """u for all 65536 bf16 patterns (non-finite ones replaced by 0) must be
    the oracle's rounding, bit for bit: this exercises the fp64 recomputation
    near bf16 ties, the subnormal range and the exp overflow region."""
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    allb[(allb & 0x7F80) == 0x7F80] = 0
    B, D = 16, 4096
    temb = allb.reshape(B, D)
    W = np.zeros((2 * D, D), np.uint16)
    b = np.zeros(2 * D, np.uint16)
    _, u = binding.adaln_proj_fwd(dev_bf16(temb), dev_bf16(W), dev_bf16(b))
    assert_bitwise(host_bf16(u), oracle.silu_bf16(temb), "silu over all bf16")


@pytest.mark.parametrize("B,D", [(2, 4096), (2, 3072), (1, 3072)])
def test_silu_every_bf16_input_small_batch(B, D):
    """The same 65536 patterns through the one- and two-sample projection
    (the streaming kernel, and D = 4096 beyond its register budget): u bit
    for bit, and emb = bf16(bias) exactly when W is zero."""
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    allb[(allb & 0x7F80) == 0x7F80] = 0
    n = B * D
    chunks = (allb.size + n - 1) // n
    padded = np.zeros(chunks * n, np.uint16)
    padded[:allb.size] = allb
    W = dev_bf16(np.zeros((2 * D, D), np.uint16))
    bias = np.arange(2 * D, dtype=np.uint16) % 0x3F00
    bd = dev_bf16(bias)
    for c in range(chunks):
        temb = padded[c * n:(c + 1) * n].reshape(B, D)
        emb, u = binding.adaln_proj_fwd(dev_bf16(temb), W, bd)
        assert_bitwise(host_bf16(u), oracle.silu_bf16(temb), f"silu chunk {c}")
        assert_bitwise(host_bf16(emb), np.broadcast_to(bias, (B, 2 * D)), f"emb chunk {c}")


def test_proj_fwd_weight_zero_gives_bias():
    inp = synth.make_inputs(3, 1, 3072, 7)
    emb, _ = binding.adaln_proj_fwd(dev_bf16(inp["temb"]), dev_bf16(np.zeros_like(inp["W"])), dev_bf16(inp["b"]))
    assert_bitwise(host_bf16(emb), np.broadcast_to(inp["b"], (3, 6144)).astype(np.uint16), "W=0")


# ---------------------------------------------------------------------------
# LayerNorm + modulation forward
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("B,S,D,seed,outl", [(2, 33, 3072, 0, 0.0), (2, 64, 3072, 1, 0.05), (1, 1, 3072, 2, 0.0),
                                             (3, 7, 256, 3, 0.0), (2, 5, 8, 4, 0.0), (2, 9, 520, 5, 0.0),
                                             (1, 3, 8192, 6, 0.0), (2, 6, 4104, 7, 0.2), (2, 9, 2056, 8, 0.0),
                                             (1, 5, 4096, 9, 0.0)])
def test_out_fwd(B, S, D, seed, outl):
    inp = synth.make_inputs(B, S, D, seed, outlier_frac=outl)
    emb = synth.normal_bf16(synth.stream_key(seed, "aux"), B * 2 * D, std=0.3).reshape(B, 2 * D)
    out, mean, rstd = binding.adaln_out_fwd(dev_bf16(inp["x"]), dev_bf16(emb))
    w_out, w_mean, w_rstd = oracle.out_fwd(inp["x"], emb)
    xf = bf16_to_f64(inp["x"])
    onep, shift = onep_shift(emb, D)
    st = check_bf16(host_bf16(out), w_out, floor_out(xf, onep, shift), what="out")
    assert st["exact"] >= 0.95 * st["n"], st
    check_f32(host_f32(mean), w_mean, F_RED * np.abs(xf).mean(-1), what="mean")
    check_f32(host_f32(rstd), w_rstd, what="rstd")


def test_out_fwd_plain_layernorm_and_constant_rows():
    D = 3072
    inp = synth.make_inputs(2, 5, D, 8)
    x = inp["x"].copy()
    x[1, 2, :] = 0x3FC0  # a constant row: xhat = 0, out = shift
    emb = np.zeros((2, 2 * D), np.uint16)
    emb[:, D:] = synth.normal_bf16(synth.stream_key(8, "aux"), 2 * D).reshape(2, D)
    out, mean, rstd = binding.adaln_out_fwd(dev_bf16(x), dev_bf16(emb))
    o = host_bf16(out)
    assert_bitwise(o[1, 2], emb[1, D:], "constant row gives shift")
    emb0 = np.zeros((2, 2 * D), np.uint16)
    out0, _, _ = binding.adaln_out_fwd(dev_bf16(x), dev_bf16(emb0))
    w0, _, _ = oracle.out_fwd(x, emb0)
    check_bf16(host_bf16(out0), w0, what="plain LN")


# ---------------------------------------------------------------------------
# backward of LayerNorm + modulation, token tree
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("B,S,D,seed,outl", [(2, 33, 3072, 0, 0.0), (1, 1, 3072, 1, 0.0), (2, 32, 3072, 2, 0.0),
                                             (2, 69, 3072, 3, 0.03), (3, 7, 256, 4, 0.0), (2, 40, 8, 5, 0.0),
                                             (1, 35, 4104, 6, 0.0), (1, 33, 8192, 7, 0.0), (1, 1100, 64, 8, 0.0),
                                             (2, 45, 2056, 9, 0.0), (2, 40, 2560, 10, 0.02), (2, 33, 2048, 11, 0.0),
                                             (1, 37, 4096, 12, 0.0)])
def test_out_bwd(B, S, D, seed, outl):
    inp = synth.make_inputs(B, S, D, seed, outlier_frac=outl)
    emb = synth.normal_bf16(synth.stream_key(seed, "aux"), B * 2 * D, std=0.3).reshape(B, 2 * D)
    x, dy = dev_bf16(inp["x"]), dev_bf16(inp["dy"])
    _, mean, rstd = binding.adaln_out_fwd(x, dev_bf16(emb))
    dx, d_emb = binding.adaln_out_bwd(dy, x, dev_bf16(emb), mean, rstd)
    torch.cuda.synchronize()
    w_dx, w_demb = oracle.out_bwd(inp["dy"], inp["x"], emb)
    xf, gf = bf16_to_f64(inp["x"]), bf16_to_f64(inp["dy"])
    onep, _ = onep_shift(emb, D)
    st = check_bf16(host_bf16(dx), w_dx, floor_dx(xf, gf, onep), what="dx")
    assert st["exact"] >= 0.9 * st["n"], st
    check_f32(host_f32(d_emb), w_demb, floor_d_emb(xf, gf), what="d_emb")
    # staged, bit for bit: the tree over the products formed from the GPU's row statistics
    prod = oracle.bwd_products_f32(inp["dy"], inp["x"], host_f32(mean), host_f32(rstd))
    assert_bitwise(host_f32(d_emb), oracle.token_tree_f32(prod), "d_emb vs fp32 tree replay")
    # the fused tree and the standalone tree agree byte for byte on the same products
    assert_bitwise(host_f32(d_emb), host_f32(binding.token_sum_tree(dev_f32(prod))), "fused vs token_sum_tree")


def test_out_bwd_empty_sequence_writes_zeros():
    D = 256
    x = torch.zeros((2, 0, D), dtype=torch.bfloat16, device="cuda")
    emb = dev_bf16(np.zeros((2, 2 * D), np.uint16))
    mean = torch.zeros((2, 0), device="cuda")
    d_emb = torch.full((2, 2 * D), float("nan"), device="cuda")
    dx, d_emb = binding.adaln_out_bwd(x, x, emb, mean, mean, d_emb=d_emb)
    assert torch.all(d_emb == 0) and not torch.any(torch.signbit(d_emb))


@pytest.mark.parametrize("S", [1, 2, 31, 32, 33, 63, 64, 65, 1000, 1024, 1025, 4096, 6032, 6889, 33000, 40000])
def test_token_sum_tree_bitwise(S):
    B, H = 2, 20
    key = synth.stream_key(S, "aux")
    a = (synth.normal(key, B * S * H) * np.exp2(np.round(synth.normal(key, B * S * H, start=B * S * H) * 4)))
    a = a.astype(np.float32).reshape(B, S, H)
    got = host_f32(binding.token_sum_tree(dev_f32(a)))
    assert_bitwise(got, oracle.token_tree_f32(a), f"tree S={S}")
    exact = oracle.token_sum_f64(a)
    bound = 2.0 ** -23 * np.abs(exact) + 2.0 ** -30 * np.abs(a.astype(np.float64)).sum(1)
    assert np.all(np.abs(got - exact) <= bound)


def test_token_sum_tree_cancellation_worked_example():
    S = 6032
    cases = [(0, 11), (0, 1), (0, 31), (31, 32), (5, 40), (100, 5000), (3000, 3001), (6030, 6031), (0, 6031), (6031, 0)]
    a = np.ones((len(cases), S, 4), np.float32)
    for i, (p, m) in enumerate(cases):
        a[i, p, :] = 2.0 ** 26
        a[i, m, :] = -(2.0 ** 26)
    got = host_f32(binding.token_sum_tree(dev_f32(a)))
    assert np.all(got == 6030.0), got[:, 0]


def test_token_sum_tree_output_is_fresh_for_one_token():
    a = dev_f32(np.arange(12, dtype=np.float32).reshape(1, 1, 12))
    out = binding.token_sum_tree(a)
    assert out.data_ptr() != a.data_ptr()
    assert_bitwise(host_f32(out), host_f32(a)[:, 0, :], "S=1")


# ---------------------------------------------------------------------------
# projection backward
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("B,D,seed", [(2, 3072, 0), (1, 3072, 1), (4, 3072, 2), (5, 3072, 3), (64, 512, 4),
                                      (3, 8, 5), (37, 1024, 6), (2, 4104, 7), (3, 3072, 8), (1, 256, 9)])
def test_proj_bwd(B, D, seed):
    """One pass over W for B <= 4: the whole-slab form where D % 256 == 0 and B
    fills the sample chunk (B = 1, 2, 4), the general form otherwise (B = 3,
    D = 8 or 4104); the tiled dW kernels for B > 4."""
    inp = synth.make_inputs(B, 1, D, seed)
    d_emb = (synth.normal(synth.stream_key(seed, "aux"), B * 2 * D) * 4).astype(np.float32).reshape(B, 2 * D)
    temb, W = dev_bf16(inp["temb"]), dev_bf16(inp["W"])
    _, u = binding.adaln_proj_fwd(temb, W, dev_bf16(inp["b"]))
    N = 2 * D
    dW = torch.empty((N, D), dtype=torch.bfloat16, device="cuda")
    db = torch.empty((N,), dtype=torch.bfloat16, device="cuda")
    dW_acc = torch.empty((N, D), device="cuda")
    db_acc = torch.empty((N,), device="cuda")
    d_temb, dW_acc, db_acc, dW, db = binding.adaln_proj_bwd(dev_f32(d_emb), temb, u, W, dW_acc=dW_acc,
                                                            db_acc=db_acc, dW=dW, db=db)
    torch.cuda.synchronize()
    w_dt, w_dW, w_db = oracle.proj_bwd(d_emb, inp["temb"], inp["W"])
    e = bf16_to_f64(synth.bf16_bits_from_f32(d_emb))
    t = bf16_to_f64(inp["temb"])
    fl = floor_d_temb(e, bf16_to_f64(inp["W"]), oracle.dsilu_f64(t))
    st = check_bf16(host_bf16(d_temb), w_dt, fl, what="d_temb")
    assert st["exact"] >= 0.95 * st["n"], st
    s_dW, s_db = oracle.wgrad_seq_f32(d_emb, inp["temb"])
    assert_bitwise(host_f32(dW_acc), s_dW, "dW_acc vs sequential replay")
    assert_bitwise(host_f32(db_acc), s_db, "db_acc vs sequential replay")
    assert_bitwise(host_bf16(dW), synth.bf16_bits_from_f32(s_dW), "dW = bf16(acc)")
    assert_bitwise(host_bf16(db), synth.bf16_bits_from_f32(s_db), "db = bf16(acc)")
    check_f32(s_dW, w_dW, (B + 1) * 2.0 ** -24 * (np.abs(e).T @ np.abs(bf16_to_f64(oracle.silu_bf16(inp["temb"])))),
              what="dW vs fp64")


@pytest.mark.parametrize("B,D,split", [(2, 3072, 1), (6, 512, 2), (12, 256, 5)])
def test_proj_bwd_accumulate_over_calls(B, D, split):
    """Samples 0..k-1 then k..B-1 with accumulate = 1 give the bytes of one call."""
    inp = synth.make_inputs(B, 1, D, 11)
    d_emb = synth.normal(synth.stream_key(11, "aux"), B * 2 * D).astype(np.float32).reshape(B, 2 * D)
    temb, W = dev_bf16(inp["temb"]), dev_bf16(inp["W"])
    _, u = binding.adaln_proj_fwd(temb, W, dev_bf16(inp["b"]))
    N = 2 * D
    accW = torch.empty((N, D), device="cuda")
    accb = torch.empty((N,), device="cuda")
    binding.adaln_proj_bwd(dev_f32(d_emb), temb, u, W, dW_acc=accW, db_acc=accb)
    one = host_f32(accW), host_f32(accb)
    cW = torch.empty((N, D), device="cuda")
    cb = torch.empty((N,), device="cuda")
    for i, j in [(0, split), (split, B)]:
        binding.adaln_proj_bwd(dev_f32(d_emb[i:j]), temb[i:j], u[i:j], W, dW_acc=cW, db_acc=cb, accumulate=i > 0)
    assert_bitwise(host_f32(cW), one[0], "chunked dW")
    assert_bitwise(host_f32(cb), one[1], "chunked db")
    # appending zero samples changes nothing
    z = torch.zeros((3, 2 * D), device="cuda")
    binding.adaln_proj_bwd(z, temb[:1].repeat(3, 1), u[:1].repeat(3, 1), W, dW_acc=cW, db_acc=cb, accumulate=True)
    assert_bitwise(host_f32(cW), one[0], "zero padding")


def test_proj_bwd_no_samples_overwrite_writes_zeros():
    D = 64
    W = dev_bf16(synth.make_inputs(1, 1, D, 0)["W"])
    e = torch.zeros((0, 2 * D), device="cuda")
    t = torch.zeros((0, D), dtype=torch.bfloat16, device="cuda")
    accW = torch.full((2 * D, D), 7.0, device="cuda")
    accb = torch.full((2 * D,), 7.0, device="cuda")
    binding.adaln_proj_bwd(e, t, t, W, dW_acc=accW, db_acc=accb)
    assert torch.all(accW == 0) and torch.all(accb == 0)


# ---------------------------------------------------------------------------
# the whole step, end to end, against the oracle's chain
# ---------------------------------------------------------------------------

def test_end_to_end_small_config():
    """B=2, S=33, D=3072, seed 0: the chain through all four entry points.
    Each stage is compared with the oracle given the GPU's previous stage."""
    from gpu_util import run_step
    inp = synth.make_inputs(2, 33, 3072, 0)
    r = run_step(to_device(inp))
    torch.cuda.synchronize()
    emb = host_bf16(r["emb"])
    fl = floor_emb(bf16_to_f64(oracle.silu_bf16(inp["temb"])), bf16_to_f64(inp["W"]), bf16_to_f64(inp["b"]))
    check_bf16(emb, oracle.proj_fwd(inp["temb"], inp["W"], inp["b"]), fl, what="emb")
    w_out, _, _ = oracle.out_fwd(inp["x"], emb)
    check_bf16(host_bf16(r["out"]), w_out, floor_out(bf16_to_f64(inp["x"]), *onep_shift(emb, 3072)), what="out")
    w_dx, w_demb = oracle.out_bwd(inp["dy"], inp["x"], emb)
    xf, gf = bf16_to_f64(inp["x"]), bf16_to_f64(inp["dy"])
    check_bf16(host_bf16(r["dx"]), w_dx, floor_dx(xf, gf, onep_shift(emb, 3072)[0]), what="dx")
    check_f32(host_f32(r["d_emb"]), w_demb, floor_d_emb(xf, gf), what="d_emb")
    d_emb = host_f32(r["d_emb"])
    w_dt, _, _ = oracle.proj_bwd(d_emb, inp["temb"], inp["W"], want_dW=False)
    check_bf16(host_bf16(r["d_temb"]), w_dt, what="d_temb", floor=floor_d_temb(
        bf16_to_f64(synth.bf16_bits_from_f32(d_emb)), bf16_to_f64(inp["W"]), oracle.dsilu_f64(bf16_to_f64(inp["temb"]))))
    s_dW, s_db = oracle.wgrad_seq_f32(d_emb, inp["temb"])
    assert_bitwise(host_bf16(r["dW"]), synth.bf16_bits_from_f32(s_dW), "dW")
    assert_bitwise(host_bf16(r["db"]), synth.bf16_bits_from_f32(s_db), "db")


@pytest.mark.parametrize("B,D", [(2, 3072), (6, 512), (3, 64)])
def test_proj_wgrad_rows_equals_rows_of_proj_bwd(B, D):
    """The row blocks of adaln_proj_wgrad_rows (the sharded step's weight
    gradient), concatenated, are adaln_proj_bwd's dW and db bit for bit: with
    one and with several samples per call, fp32 accumulators and bf16 outputs,
    overwrite and accumulate."""
    lib()
    inp = synth.make_inputs(B, 1, D, 11)
    temb, W = dev_bf16(inp["temb"]), dev_bf16(inp["W"])
    N = 2 * D
    d_emb = dev_f32(synth.normal(synth.stream_key(11, "aux"), B * N).astype(np.float32).reshape(B, N) * 2)
    u = dev_bf16(oracle.silu_bf16(inp["temb"]))
    acc0 = dev_f32(synth.normal(synth.stream_key(12, "aux"), N * D).astype(np.float32).reshape(N, D))
    accb0 = dev_f32(synth.normal(synth.stream_key(13, "aux"), N).astype(np.float32))
    for accumulate in (False, True):
        refW = acc0.clone()
        refb = accb0.clone()
        dW = torch.empty((N, D), dtype=torch.bfloat16, device="cuda")
        db = torch.empty((N,), dtype=torch.bfloat16, device="cuda")
        binding.adaln_proj_bwd(d_emb, temb, u, W, dW_acc=refW, db_acc=refb, dW=dW, db=db, accumulate=accumulate)
        cuts = [0, N // 3, N // 3 + 8, 2 * N // 3, N]
        parts = []
        for n0, n1 in zip(cuts[:-1], cuts[1:]):
            a = acc0[n0:n1].clone()
            ab = accb0[n0:n1].clone()
            rW = torch.empty((n1 - n0, D), dtype=torch.bfloat16, device="cuda")
            rb = torch.empty((n1 - n0,), dtype=torch.bfloat16, device="cuda")
            binding.adaln_proj_wgrad_rows(d_emb, u, n0, n1, dW_acc=a, db_acc=ab, dW=rW, db=rb, accumulate=accumulate)
            parts.append((a, ab, rW, rb))
        torch.cuda.synchronize()
        for i, (ref, name) in enumerate(((refW, "dW_acc"), (refb, "db_acc"), (dW, "dW"), (db, "db"))):
            got = torch.cat([p[i] for p in parts])
            assert_bitwise(host_f32(got) if got.dtype == torch.float32 else host_bf16(got),
                           host_f32(ref) if ref.dtype == torch.float32 else host_bf16(ref), f"{name} acc={accumulate}")
    assert binding.device_error() == 0


def test_sharded_step_on_one_gpu_matches_the_step():
    """The sharded step through the library with one rank (no exchange): its
    per-sample results and its whole row block of dW, db are the plain step's
    bytes."""
    from invariant_dit_adaln_gb300 import sharded
    from gpu_util import run_step
    lib()
    B, S, D = 3, 40, 512
    inp = to_device(synth.make_inputs(B, S, D, 14, outlier_frac=0.05))
    ref = run_step(inp)
    plan = sharded.ShardPlan.make(B, D, 1, 0)
    got = sharded.sharded_step(inp["x"], inp["dy"], inp["temb"], inp["W"], inp["b"], plan, dist=None)
    torch.cuda.synchronize()
    for k in ("emb", "u", "out", "mean", "rstd", "dx", "d_emb", "d_temb"):
        assert torch.equal(got[k].view(torch.uint8), ref[k].view(torch.uint8)), k
    assert torch.equal(got["dW_rows"].view(torch.int16), ref["dW"].view(torch.int16))
    assert torch.equal(got["db_rows"].view(torch.int16), ref["db"].view(torch.int16))
    assert binding.device_error() == 0
