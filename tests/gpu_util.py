"""Helpers for the GPU tests: moving bf16 bit patterns between numpy and torch,
and running the operator through the C ABI binding."""

from __future__ import annotations

import numpy as np
import torch

from invariant_dit_adaln_gb300 import binding, build


def lib():
    build.build()
    return binding.load()


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 patterns -> CUDA bfloat16 tensor (same bits)."""
    a = np.ascontiguousarray(bits, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)


def host_bf16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy()


def run_forward(inp, eps=1e-6):
    """Device inputs dict -> (emb, u, out, mean, rstd) on the device."""
    emb, u = binding.adaln_proj_fwd(inp["temb"], inp["W"], inp["b"])
    out, mean, rstd = binding.adaln_out_fwd(inp["x"], emb, eps=eps)
    return emb, u, out, mean, rstd


def run_step(inp, eps=1e-6):
    """The whole hot path on device inputs: forward and backward.
    Returns a dict of device tensors."""
    emb, u, out, mean, rstd = run_forward(inp, eps)
    dx, d_emb = binding.adaln_out_bwd(inp["dy"], inp["x"], emb, mean, rstd)
    D = inp["x"].shape[-1]
    dW = torch.empty((2 * D, D), dtype=torch.bfloat16, device="cuda")
    db = torch.empty((2 * D,), dtype=torch.bfloat16, device="cuda")
    d_temb, _, _, dW, db = binding.adaln_proj_bwd(d_emb, inp["temb"], u, inp["W"], dW=dW, db=db)
    return {"emb": emb, "u": u, "out": out, "mean": mean, "rstd": rstd, "dx": dx, "d_emb": d_emb,
            "d_temb": d_temb, "dW": dW, "db": db}


def to_device(inputs: dict) -> dict:
    return {k: dev_bf16(v) for k, v in inputs.items() if k in ("x", "dy", "temb", "W", "b")}
