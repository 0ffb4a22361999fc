"""adaln_out_fwd_proj (the forward with proj_out on the tensor cores) against
the oracle and against adaln_out_fwd, on the GPU.

out, mean and rstd must be the bytes adaln_out_fwd gives; y is checked
against the oracle's correctly rounded projection of the GPU's own out (1 bf16
ulp or the fp32 floor 2^-16 * sum |out Wp| + |bp|), and every token's row of y
must have the same bytes at any batch size, sequence length and position.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from invariant_dit_adaln_gb300 import binding, synth
from gpu_util import dev_bf16, host_bf16, lib
from tolerance import F_OUT, bf16_to_f64, check_bf16

pytestmark = pytest.mark.gpu

J = 64


@pytest.fixture(scope="module", autouse=True)
def _lib():
    oracle.build()
    lib()
    yield
    assert binding.device_error() == 0


def _inputs(B, S, D, seed, outlier_frac=0.0):
    i = synth.make_inputs(B, S, D, seed, outlier_frac=outlier_frac)
    emb = synth.normal_bf16(synth.stream_key(seed, "aux"), B * 2 * D, std=0.3).reshape(B, 2 * D)
    Wp = synth.normal_bf16(synth.stream_key(seed, "W"), J * D, std=0.02).reshape(J, D)
    bp = synth.normal_bf16(synth.stream_key(seed, "b"), J, std=0.02)
    return i["x"], emb, Wp, bp


@pytest.mark.parametrize("B,S,D,seed,outl", [(2, 33, 3072, 0, 0.0), (1, 1, 3072, 1, 0.0), (3, 130, 1024, 2, 0.0),
                                             (2, 200, 64, 3, 0.0), (2, 300, 3072, 4, 0.05),
                                             (2, 4096, 3072, 5, 0.01)])
def test_out_fwd_proj(B, S, D, seed, outl):
    x, emb, Wp, bp = _inputs(B, S, D, seed, outl)
    xd, ed = dev_bf16(x), dev_bf16(emb)
    out, mean, rstd, y = binding.adaln_out_fwd_proj(xd, ed, dev_bf16(Wp), dev_bf16(bp))
    out2, mean2, rstd2 = binding.adaln_out_fwd(xd, ed)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(mean.view(torch.int32), mean2.view(torch.int32))
    assert torch.equal(rstd.view(torch.int32), rstd2.view(torch.int32))
    o = host_bf16(out).reshape(B * S, D)
    yg = host_bf16(y).reshape(B * S, J)
    if B * S > 2048:  # every 8th token row (the first and last tile included) at the full size
        rows = np.unique(np.concatenate([np.arange(0, B * S, 8), np.arange(B * S - 128, B * S)]))
        o, yg = o[rows], yg[rows]
    want = oracle.proj_out(o, Wp, bp)
    fl = F_OUT * (np.abs(bf16_to_f64(o)) @ np.abs(bf16_to_f64(Wp)).T + np.abs(bf16_to_f64(bp)))
    st = check_bf16(yg, want, fl, what="proj_out y")
    assert st["exact"] >= 0.99 * st["n"], st


def test_proj_out_rows_do_not_depend_on_batch_or_position():
    """y of each sample of a batch of 3 (S = 45: tiles of 128 token rows cut
    across samples) has the bytes of the sample run alone, and of the same
    tokens at another sequence length (its first 20 tokens)."""
    D = 3072
    x, emb, Wp, bp = _inputs(3, 45, D, 6)
    xd, ed, wd, bd = dev_bf16(x), dev_bf16(emb), dev_bf16(Wp), dev_bf16(bp)
    _, _, _, y = binding.adaln_out_fwd_proj(xd, ed, wd, bd)
    for b in range(3):
        _, _, _, y1 = binding.adaln_out_fwd_proj(xd[b:b + 1].contiguous(), ed[b:b + 1].contiguous(), wd, bd)
        assert torch.equal(y[b:b + 1].view(torch.int16), y1.view(torch.int16)), b
        _, _, _, y2 = binding.adaln_out_fwd_proj(xd[b:b + 1, :20].contiguous(), ed[b:b + 1].contiguous(), wd, bd)
        assert torch.equal(y[b:b + 1, :20].view(torch.int16), y2.view(torch.int16)), b
