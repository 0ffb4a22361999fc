"""Bytewise batch invariance of the whole fwd+bwd path on the GPU.

The pages' protocol (RL-Kernel PR 538, "Prior art & reuse decision"): a
singleton compared with every row of B = 64/257/2048, three seeds, B = 2 vs
B = 1 at long sequences, and a workload run in five chunkings.  Every per-sample
output (emb, u, out, mean, rstd, dx, d_emb, d_temb) of sample b in a batch
must have the bytes of the same sample run alone; dW and db summed over a
workload in chunks (accumulating into fp32) must have the bytes of one call.
"""

from __future__ import annotations

import pytest
import torch

from invariant_dit_adaln_gb300 import binding
from gpu_util import lib, run_step

pytestmark = pytest.mark.gpu

PER_SAMPLE = ("emb", "u", "out", "mean", "rstd", "dx", "d_emb", "d_temb")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib()
    yield
    assert binding.device_error() == 0


def _device_inputs(n, S, D, seed, outlier_frac=0.0):
    """Seeded synthetic inputs generated on the device (these tests compare the
    GPU with itself, and the host generator would take minutes at these
    sizes): x, dy, temb ~ N(0, 1) from torch's Philox generator, rounded to
    bf16; W, b ~ N(0, 0.02^2); optionally floor(frac*n*S) token rows of x and
    dy scaled by 50 in fp32 before the rounding."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x = torch.randn((n, S, D), generator=g, device="cuda")
    dy = torch.randn((n, S, D), generator=g, device="cuda")
    k = int(outlier_frac * n * S)
    if k:
        rows = torch.randperm(n * S, generator=g, device="cuda")[:k]
        x.view(n * S, D)[rows] *= 50
        dy.view(n * S, D)[rows] *= 50
    temb = torch.randn((n, D), generator=g, device="cuda").to(torch.bfloat16)
    W = (torch.randn((2 * D, D), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    b = (torch.randn((2 * D,), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    return {"x": x.to(torch.bfloat16), "dy": dy.to(torch.bfloat16), "temb": temb, "W": W, "b": b}


def _bits(t):
    return t.contiguous().view(torch.int16 if t.element_size() == 2 else torch.int32)


def _compare_rows(batch, single, b, what):
    for k in PER_SAMPLE:
        if not torch.equal(_bits(batch[k][b:b + 1]), _bits(single[k])):
            raise AssertionError(f"{what}: {k} of sample {b} differs from the sample run alone")


def _one(dev, b):
    return {k: (v if k in ("W", "b") else v[b:b + 1]) for k, v in dev.items()}


def test_projection_is_M_invariant_across_batch_sizes():
    """emb and u rows have the same bits for every B from 1 to 4096 and for
    every position of a sample in the batch: the tensor-core tiles of 16
    samples, a ragged last tile, the u box rounded up to 8 rows below 16
    samples, one to 16 sample tiles per CTA and the stage layouts chosen by
    batch size."""
    D = 3072
    big = _device_inputs(4096, 1, D, seed=3)
    W, b = big["W"], big["b"]
    ref, uref = binding.adaln_proj_fwd(big["temb"], W, b)
    for B in [1, 2, 3, 4, 5, 7, 8, 9, 15, 16, 17, 33, 64, 80, 81, 127, 128, 129, 255, 256, 257, 1000, 2048]:
        e, u = binding.adaln_proj_fwd(big["temb"][:B], W, b)
        assert torch.equal(_bits(e), _bits(ref[:B])), B
        assert torch.equal(_bits(u), _bits(uref[:B])), B
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    for n, start in [(300, 0), (129, 3000), (2, 4094)]:
        idx = start + torch.randperm(n, generator=g, device="cuda")
        e, u = binding.adaln_proj_fwd(big["temb"][idx].contiguous(), W, b)
        assert torch.equal(_bits(e), _bits(ref[idx])), (n, start)
        assert torch.equal(_bits(u), _bits(uref[idx])), (n, start)


def test_projection_at_4096_samples_matches_the_oracle():
    """Sampled samples of the 4096-sample projection (the first and last of
    each tile of 128, and a few inside) against the oracle."""
    import numpy as np
    import oracle
    from gpu_util import host_bf16
    from tolerance import bf16_to_f64, check_bf16, floor_emb
    oracle.build()
    D = 3072
    big = _device_inputs(4096, 1, D, seed=5)
    emb, u = binding.adaln_proj_fwd(big["temb"], big["W"], big["b"])
    rows = sorted({0, 1, 127, 128, 255, 2047, 2048, 3071, 4094, 4095, 1000, 1729})
    temb = host_bf16(big["temb"])[rows]
    W, bias = host_bf16(big["W"]), host_bf16(big["b"])
    want = oracle.proj_fwd(temb, W, bias)
    u_ref = oracle.silu_bf16(temb)
    assert np.array_equal(host_bf16(u)[rows], u_ref)
    fl = floor_emb(bf16_to_f64(u_ref), bf16_to_f64(W), bf16_to_f64(bias))
    st = check_bf16(host_bf16(emb)[rows], want, fl, what="emb at B=4096")
    assert st["exact"] >= 0.99 * st["n"], st


@pytest.mark.parametrize("seed", [0, 127, 2026])
@pytest.mark.parametrize("S", [31, 32, 33])
@pytest.mark.parametrize("B", [64, 257])
def test_every_row_matches_the_singleton(B, S, seed):
    D = 3072
    dev = _device_inputs(B, S, D, seed)
    batch = run_step(dev)
    for b in range(B):
        _compare_rows(batch, run_step(_one(dev, b)), b, f"B={B} S={S} seed={seed}")
    # the weight gradient of the batch equals the samples accumulated one by one
    N = 2 * D
    accW = torch.empty((N, D), device="cuda")
    accb = torch.empty((N,), device="cuda")
    for b in range(B):
        binding.adaln_proj_bwd(batch["d_emb"][b:b + 1], dev["temb"][b:b + 1], batch["u"][b:b + 1], dev["W"],
                               dW_acc=accW, db_acc=accb, accumulate=b > 0)
    dW = torch.empty((N, D), dtype=torch.bfloat16, device="cuda")
    db = torch.empty((N,), dtype=torch.bfloat16, device="cuda")
    binding.adaln_proj_bwd(torch.zeros((0, N), device="cuda"), dev["temb"][:0], batch["u"][:0], dev["W"],
                           dW_acc=accW, db_acc=accb, dW=dW, db=db, accumulate=True)
    assert torch.equal(_bits(dW), _bits(batch["dW"]))
    assert torch.equal(_bits(db), _bits(batch["db"]))


def test_rows_of_a_2048_batch_match_the_singleton():
    B, S, D = 2048, 33, 3072
    dev = _device_inputs(B, S, D, seed=5)
    batch = run_step(dev)
    for b in [0, 1, 2, 777, 1023, 1024, 2046, 2047]:
        _compare_rows(batch, run_step(_one(dev, b)), b, "B=2048")


@pytest.mark.parametrize("S", [4096, 6032, 6889])
def test_two_samples_match_one(S):
    D = 3072
    dev = _device_inputs(2, S, D, seed=1, outlier_frac=0.01)
    batch = run_step(dev)
    for b in range(2):
        _compare_rows(batch, run_step(_one(dev, b)), b, f"B=2 vs 1, S={S}")


def test_run_to_run_determinism():
    dev = _device_inputs(2, 4096, 3072, seed=2, outlier_frac=0.01)
    r1 = run_step(dev)
    r2 = run_step(dev)
    for k in r1:
        assert torch.equal(r1[k].view(torch.uint8), r2[k].view(torch.uint8)), k


def _chunked(dev, chunk, D):
    """Runs the workload in chunks of `chunk` samples; returns per-sample
    outputs concatenated and dW/db accumulated over the chunks."""
    n = dev["x"].shape[0]
    N = 2 * D
    accW = torch.empty((N, D), device="cuda")
    accb = torch.empty((N,), device="cuda")
    outs = {k: [] for k in PER_SAMPLE}
    for i in range(0, n, chunk):
        part = {k: (v if k in ("W", "b") else v[i:i + chunk]) for k, v in dev.items()}
        emb, u = binding.adaln_proj_fwd(part["temb"], part["W"], part["b"])
        out, mean, rstd = binding.adaln_out_fwd(part["x"], emb)
        dx, d_emb = binding.adaln_out_bwd(part["dy"], part["x"], emb, mean, rstd)
        d_temb, _, _, _, _ = binding.adaln_proj_bwd(d_emb, part["temb"], u, part["W"], dW_acc=accW, db_acc=accb,
                                                    accumulate=i > 0)
        for k, v in zip(PER_SAMPLE, (emb, u, out, mean, rstd, dx, d_emb, d_temb)):
            outs[k].append(v)
    return {k: torch.cat(v) for k, v in outs.items()}, accW, accb


@pytest.mark.parametrize("n,chunks", [(256, [256, 128, 16, 4, 1])])
def test_chunking_invariance(n, chunks):
    """The chunking workload (samples of S=256) at 256 samples, in five
    chunkings: every output and dW/db byte-identical."""
    D, S = 3072, 256
    dev = _device_inputs(n, S, D, seed=4)
    ref, refW, refb = _chunked(dev, chunks[0], D)
    for c in chunks[1:]:
        got, gW, gb = _chunked(dev, c, D)
        for k in PER_SAMPLE:
            assert torch.equal(got[k].view(torch.uint8), ref[k].view(torch.uint8)), (c, k)
        assert torch.equal(gW.view(torch.int32), refW.view(torch.int32)), c
        assert torch.equal(gb.view(torch.int32), refb.view(torch.int32)), c


def _oracle_check_samples(dev, ref, refW, refb, samples, rows, D):
    """The 1 x n chunk against the oracle: every per-sample output of the
    listed samples, and the listed rows of dW, db summed over all n samples
    (the chunked projection and the tiled weight-gradient kernels run only at
    batches this large)."""
    import numpy as np
    import oracle
    from gpu_util import host_bf16, host_f32
    from tolerance import (assert_bitwise, bf16_to_f64, check_bf16, check_f32, check_rows, floor_d_emb,
                           floor_d_temb, floor_emb)
    oracle.build()
    idx = torch.tensor(samples, device="cuda")
    h = {k: host_bf16(dev[k].index_select(0, idx)) for k in ("x", "dy", "temb")}
    W, b = host_bf16(dev["W"]), host_bf16(dev["b"])
    g = {k: (host_bf16(v.index_select(0, idx)) if v.dtype == torch.bfloat16 else host_f32(v.index_select(0, idx)))
         for k, v in ref.items()}
    u_ref = oracle.silu_bf16(h["temb"])
    check_bf16(g["emb"], oracle.proj_fwd(h["temb"], W, b), floor_emb(bf16_to_f64(u_ref), bf16_to_f64(W), bf16_to_f64(b)),
               what="1x4096 chunk: emb of sampled samples")
    assert_bitwise(g["u"], u_ref, "1x4096 chunk: u")
    check_rows(h["x"], h["dy"], g["emb"], g, oracle, what="1x4096 chunk: sampled samples")
    prod = oracle.bwd_products_f32(h["dy"], h["x"], g["mean"], g["rstd"])
    assert_bitwise(g["d_emb"], oracle.token_tree_f32(prod), "1x4096 chunk: d_emb vs the fp32 tree")
    _, w_demb = oracle.out_bwd(h["dy"], h["x"], g["emb"])
    check_f32(g["d_emb"], w_demb, floor_d_emb(bf16_to_f64(h["x"]), bf16_to_f64(h["dy"])), what="1x4096 chunk: d_emb")
    w_dt, _, _ = oracle.proj_bwd(g["d_emb"], h["temb"], W, want_dW=False)
    from invariant_dit_adaln_gb300 import synth
    fl = floor_d_temb(bf16_to_f64(synth.bf16_bits_from_f32(g["d_emb"])), bf16_to_f64(W),
                      oracle.dsilu_f64(bf16_to_f64(h["temb"])))
    check_bf16(g["d_temb"], w_dt, fl, what="1x4096 chunk: d_temb")
    sW, sb = oracle.wgrad_seq_f32_rows(host_f32(ref["d_emb"]), host_bf16(dev["temb"]), np.array(rows, np.int32))
    assert_bitwise(host_f32(refW)[rows], sW, "1x4096 chunk: sampled rows of dW")
    assert_bitwise(host_f32(refb)[rows], sb, "1x4096 chunk: sampled rows of db")


@pytest.mark.slow
def test_chunking_invariance_full_workload():
    """4096 samples of S=256 as 1x4096, 2x2048, 16x256, 64x64 and 4096x1; the
    1x4096 chunk also against the oracle on 8 samples and 16 rows of dW."""
    D, S, n = 3072, 256, 4096
    dev = _device_inputs(n, S, D, seed=6)
    ref, refW, refb = _chunked(dev, 4096, D)
    _oracle_check_samples(dev, ref, refW, refb, samples=[0, 1, 977, 2048, 2049, 3333, 4094, 4095],
                          rows=[0, 1, 255, 256, 1000, 3071, 3072, 3073, 4095, 4096, 5000, 6000, 6142, 6143, 77, 2222],
                          D=D)
    for c in [2048, 256, 64, 1]:
        got, gW, gb = _chunked(dev, c, D)
        for k in PER_SAMPLE:
            assert torch.equal(got[k].view(torch.uint8), ref[k].view(torch.uint8)), (c, k)
        assert torch.equal(gW.view(torch.int32), refW.view(torch.int32)), c
        assert torch.equal(gb.view(torch.int32), refb.view(torch.int32)), c
        del got
