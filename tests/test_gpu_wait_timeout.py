"""The time-out path of the kernels' waits, run on the GPU without a fault.

Kernels that wait on their own bulk copies give each wait a time limit; a wait
that runs out sets the library's device error word and the kernel drains the
copies it issued, then returns.  A test build of the library sends the first
wait of every waiting kernel to an mbarrier that nothing ever arrives on (a
200 us limit), so the path runs: the forward (also the block-level norm's)
reports 0x101, the backward 0x201,
the tensor-core projection 0x302 and proj_out 0x303 (the MMA thread gives up,
the TMA thread stops and lets its copies land, the cluster writes nothing and
frees its tensor memory), no drain runs out (the 0x8000 bit stays clear), and the GPU context
stays usable, shown by the release library's results afterwards being the same
bytes as before.
"""

from __future__ import annotations

import ctypes

import pytest
import torch

from invariant_dit_adaln_gb300 import binding, build, synth
from gpu_util import run_step, to_device

pytestmark = pytest.mark.gpu

FWD_WAIT, BWD_WAIT, PROJ_TC_WAIT, DRAIN_FAILED = 0x101, 0x201, 0x302, 0x8000


@pytest.fixture(scope="module")
def wait_lib():
    path = build.build(extra_flags=build.WAIT_TEST_FLAGS, variant="waittest")
    L = ctypes.CDLL(path)
    P, I = ctypes.c_void_p, ctypes.c_int
    L.adaln_out_fwd.argtypes = [P, P, P, P, P, I, I, I, ctypes.c_float, P]
    L.adaln_out_bwd.argtypes = [P, P, P, P, P, P, P, P, ctypes.c_size_t, I, I, I, P]
    L.adaln_proj_fwd.argtypes = [P, P, P, P, P, I, I, P]
    L.adaln_out_fwd_proj.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, ctypes.c_float, P]
    L.adaln_scale_residual_norm_fwd.argtypes = [P] * 8 + [I, I, I, ctypes.c_float, P]
    L.adaln_device_error.restype = I
    return L


def _bits(t):
    return t.contiguous().view(torch.int16 if t.element_size() == 2 else torch.int32)


@pytest.mark.parametrize("B,S,D", [(2, 100, 3072), (1, 40, 8192)])
def test_waits_that_run_out_report_and_return(wait_lib, B, S, D):
    L = wait_lib
    binding.load()
    inp = to_device(synth.make_inputs(B, S, D, 3, outlier_frac=0.01))
    before = run_step(inp)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    emb = before["emb"]
    out = torch.empty_like(inp["x"])
    mean = torch.empty((B, S), dtype=torch.float32, device="cuda")
    rstd = torch.empty_like(mean)
    st = torch.cuda.current_stream().cuda_stream
    assert L.adaln_out_fwd(inp["x"].data_ptr(), emb.data_ptr(), out.data_ptr(), mean.data_ptr(), rstd.data_ptr(),
                           B, S, D, 1e-6, st) == 0
    err = L.adaln_device_error()
    assert err & ~DRAIN_FAILED == FWD_WAIT and not err & DRAIN_FAILED, hex(err)
    dx = torch.empty_like(inp["x"])
    d_emb = torch.empty((B, 2 * D), dtype=torch.float32, device="cuda")
    ws = torch.empty(binding.adaln_out_bwd_workspace_bytes(B, S, D), dtype=torch.uint8, device="cuda")
    assert L.adaln_out_bwd(inp["dy"].data_ptr(), inp["x"].data_ptr(), emb.data_ptr(), before["mean"].data_ptr(),
                           before["rstd"].data_ptr(), dx.data_ptr(), d_emb.data_ptr(), ws.data_ptr(), ws.numel(),
                           B, S, D, st) == 0
    err = L.adaln_device_error()
    assert err & ~DRAIN_FAILED == BWD_WAIT and not err & DRAIN_FAILED, hex(err)
    e2 = torch.empty_like(emb)
    u2 = torch.empty_like(before["u"])
    assert L.adaln_proj_fwd(inp["temb"].data_ptr(), inp["W"].data_ptr(), inp["b"].data_ptr(), e2.data_ptr(),
                            u2.data_ptr(), B, D, st) == 0
    err = L.adaln_device_error()
    assert err & ~DRAIN_FAILED == PROJ_TC_WAIT and not err & DRAIN_FAILED, hex(err)
    # the fused forward: both kernels give up; the LayerNorm kernel's code is
    # reported first, and no drain of either ran out
    Wp = torch.zeros((64, D), dtype=torch.bfloat16, device="cuda")
    bp = torch.zeros((64,), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((B, S, 64), dtype=torch.bfloat16, device="cuda")
    assert L.adaln_out_fwd_proj(inp["x"].data_ptr(), emb.data_ptr(), Wp.data_ptr(), bp.data_ptr(), out.data_ptr(),
                                mean.data_ptr(), rstd.data_ptr(), y.data_ptr(), B, S, D, 64, 1e-6, st) == 0
    err = L.adaln_device_error()
    assert err & ~DRAIN_FAILED == FWD_WAIT and not err & DRAIN_FAILED, hex(err)
    # the block-level norm's forward (the gated residual formed in the LayerNorm kernel where D <= 4096)
    gate = torch.zeros((B, D), dtype=torch.bfloat16, device="cuda")
    r = torch.empty_like(inp["x"])
    assert L.adaln_scale_residual_norm_fwd(inp["x"].data_ptr(), inp["dy"].data_ptr(), gate.data_ptr(), emb.data_ptr(),
                                           r.data_ptr(), out.data_ptr(), mean.data_ptr(), rstd.data_ptr(), B, S, D,
                                           1e-6, st) == 0
    err = L.adaln_device_error()
    assert err & ~DRAIN_FAILED == FWD_WAIT and not err & DRAIN_FAILED, hex(err)
    assert L.adaln_device_error() == 0  # read and cleared
    # the context is still usable: the release library gives the same bytes
    after = run_step(inp)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    for k, v in before.items():
        assert torch.equal(_bits(after[k]), _bits(v)), k
