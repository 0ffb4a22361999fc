"""ctypes binding of libadaln.so: the C ABI of include/adaln.h with the same
entry-point names, taking PyTorch CUDA tensors.

This layer only marshals arguments: it checks dtypes, devices and shapes,
allocates missing outputs and workspaces with PyTorch's allocator, copies an
input whose storage offset breaks 16-byte alignment (the C ABI requires
aligned pointers), passes raw pointers and the current stream, and raises on a
non-zero status.  All computation runs in the library's CUDA kernels; there is
no fallback path.  If the library is missing, every call raises.
"""

from __future__ import annotations

import ctypes
import os
import re

import torch

from . import build as _build

_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_F = ctypes.c_float

_SIGNATURES = {
    "adaln_status_string": (ctypes.c_char_p, [_I]),
    "adaln_version": (_I, []),
    "adaln_proj_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _P]),
    "adaln_out_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _F, _P]),
    "adaln_out_bwd_workspace_bytes": (_SZ, [_I, _I, _I]),
    "adaln_out_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I, _I, _I, _P]),
    "adaln_out_bwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P]),
    "token_sum_tree_workspace_bytes": (_SZ, [_I, _I, _I]),
    "token_sum_tree": (_I, [_P, _P, _I, _I, _I, _P, _SZ, _P]),
    "adaln_proj_bwd_workspace_bytes": (_SZ, [_I, _I]),
    "adaln_proj_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _SZ, _I, _I, _P]),
    "adaln_proj_wgrad_rows": (_I, [_P, _P, _I, _I, _P, _P, _P, _P, _I, _I, _I, _P]),
    "adaln_scale_residual_norm_fwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _F, _P]),
    "adaln_scale_residual_norm_bwd_workspace_bytes": (_SZ, [_I, _I, _I]),
    "adaln_scale_residual_norm_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I, _I, _I,
                                           _P]),
    "adaln_f32_proj_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _P]),
    "adaln_f32_out_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _F, _P]),
    "adaln_f32_out_bwd_workspace_bytes": (_SZ, [_I, _I, _I]),
    "adaln_f32_out_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I, _I, _I, _P]),
    "adaln_f32_proj_bwd_workspace_bytes": (_SZ, [_I, _I]),
    "adaln_f32_proj_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _P, _SZ, _I, _I, _P]),
    "adaln_out_fwd_proj": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _P]),
    "adaln_device_error": (_I, []),
}

_lib = None


class AdaLNError(RuntimeError):
    def __init__(self, name, status):
        self.status = status
        super().__init__(f"{name} failed: {status_string(status)}")


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load libadaln.so (once) and declare its signatures.  Raises if missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first (invariant_dit_adaln_gb300.build.build()); "
                           "there is no fallback implementation")
    L = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def declared_symbols(header: str | None = None) -> list[str]:
    """Names of the functions include/adaln.h declares."""
    header = header or os.path.join(_build.INCLUDE, "adaln.h")
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)


def status_string(status: int) -> str:
    return load().adaln_status_string(int(status)).decode()


def version() -> int:
    return load().adaln_version()


def device_error() -> int:
    return load().adaln_device_error()


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------

def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _input(t: torch.Tensor, dtype, shape, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name}: expected a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous() or t.data_ptr() % 16:
        t = t.contiguous() if not t.is_contiguous() else t.clone()  # fresh, aligned storage
    return t


def _output(t, dtype, shape, name, device, zero=False):
    if t is None:
        return (torch.zeros if zero else torch.empty)(shape, dtype=dtype, device=device)
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != dtype or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected a CUDA {dtype} tensor of shape {tuple(shape)}")
    if not t.is_contiguous() or t.data_ptr() % 16:
        raise ValueError(f"{name}: outputs must be contiguous and 16-byte aligned")
    return t


def _workspace(ws, need, device):
    if need == 0:
        return None, 0
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=device)
    if ws.numel() * ws.element_size() < need:
        raise ValueError(f"workspace: {need} bytes needed")
    return ws, ws.numel() * ws.element_size()


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check(name, status):
    if status != 0:
        raise AdaLNError(name, status)


# ---------------------------------------------------------------------------
# entry points (same names as the C ABI)
# ---------------------------------------------------------------------------

def adaln_proj_fwd(temb, W, bias, emb=None, u=None, stream=None):
    """emb [B, 2D] bf16 = bf16(bf16(silu(temb)) @ W^T + bias); u = bf16(silu(temb)).
    Returns (emb, u)."""
    L = load()
    B, D = temb.shape
    temb = _input(temb, torch.bfloat16, (B, D), "temb")
    W = _input(W, torch.bfloat16, (2 * D, D), "W")
    bias = _input(bias, torch.bfloat16, (2 * D,), "bias")
    emb = _output(emb, torch.bfloat16, (B, 2 * D), "emb", temb.device)
    u = _output(u, torch.bfloat16, (B, D), "u", temb.device)
    _check("adaln_proj_fwd", L.adaln_proj_fwd(_ptr(temb), _ptr(W), _ptr(bias), _ptr(emb), _ptr(u), B, D,
                                              _stream(stream)))
    return emb, u


def adaln_out_fwd(x, emb, out=None, mean=None, rstd=None, eps=1e-6, stream=None):
    """LayerNorm(x) * (1 + scale) + shift with the autocast rounding points.
    Returns (out [B,S,D] bf16, mean [B,S] fp32, rstd [B,S] fp32)."""
    L = load()
    B, S, D = x.shape
    x = _input(x, torch.bfloat16, (B, S, D), "x")
    emb = _input(emb, torch.bfloat16, (B, 2 * D), "emb")
    out = _output(out, torch.bfloat16, (B, S, D), "out", x.device)
    mean = _output(mean, torch.float32, (B, S), "mean", x.device)
    rstd = _output(rstd, torch.float32, (B, S), "rstd", x.device)
    _check("adaln_out_fwd", L.adaln_out_fwd(_ptr(x), _ptr(emb), _ptr(out), _ptr(mean), _ptr(rstd), B, S, D,
                                            float(eps), _stream(stream)))
    return out, mean, rstd


def adaln_out_bwd_workspace_bytes(B, S, D):
    return load().adaln_out_bwd_workspace_bytes(B, S, D)


def adaln_out_bwd(dy, x, emb, mean, rstd, dx=None, d_emb=None, workspace=None, stream=None):
    """Backward of adaln_out_fwd.  Returns (dx [B,S,D] bf16, d_emb [B,2D] fp32)."""
    L = load()
    B, S, D = x.shape
    dy = _input(dy, torch.bfloat16, (B, S, D), "dy")
    x = _input(x, torch.bfloat16, (B, S, D), "x")
    emb = _input(emb, torch.bfloat16, (B, 2 * D), "emb")
    mean = _input(mean, torch.float32, (B, S), "mean")
    rstd = _input(rstd, torch.float32, (B, S), "rstd")
    dx = _output(dx, torch.bfloat16, (B, S, D), "dx", x.device)
    d_emb = _output(d_emb, torch.float32, (B, 2 * D), "d_emb", x.device)
    ws, nws = _workspace(workspace, L.adaln_out_bwd_workspace_bytes(B, S, D), x.device)
    _check("adaln_out_bwd", L.adaln_out_bwd(_ptr(dy), _ptr(x), _ptr(emb), _ptr(mean), _ptr(rstd), _ptr(dx),
                                            _ptr(d_emb), _ptr(ws), nws, B, S, D, _stream(stream)))
    return dx, d_emb


def adaln_out_fwd_proj(x, emb, Wp, bp, out=None, mean=None, rstd=None, y=None, eps=1e-6, stream=None):
    """LayerNorm + modulation forward, then proj_out: y = bf16(out Wp^T + bp)
    on the tensor cores.  Returns (out, mean, rstd, y)."""
    L = load()
    B, S, D = x.shape
    J = Wp.shape[0]
    x = _input(x, torch.bfloat16, (B, S, D), "x")
    emb = _input(emb, torch.bfloat16, (B, 2 * D), "emb")
    Wp = _input(Wp, torch.bfloat16, (J, D), "Wp")
    bp = _input(bp, torch.bfloat16, (J,), "bp")
    out = _output(out, torch.bfloat16, (B, S, D), "out", x.device)
    mean = _output(mean, torch.float32, (B, S), "mean", x.device)
    rstd = _output(rstd, torch.float32, (B, S), "rstd", x.device)
    y = _output(y, torch.bfloat16, (B, S, J), "y", x.device)
    _check("adaln_out_fwd_proj", L.adaln_out_fwd_proj(_ptr(x), _ptr(emb), _ptr(Wp), _ptr(bp), _ptr(out), _ptr(mean),
                                                      _ptr(rstd), _ptr(y), B, S, D, J, float(eps), _stream(stream)))
    return out, mean, rstd, y


def adaln_f32_proj_fwd(temb, W, bias, emb=None, u=None, stream=None):
    """fp32 projection: (emb [B,2D], u [B,D]), both fp32."""
    L = load()
    B, D = temb.shape
    temb = _input(temb, torch.float32, (B, D), "temb")
    W = _input(W, torch.float32, (2 * D, D), "W")
    bias = _input(bias, torch.float32, (2 * D,), "bias")
    emb = _output(emb, torch.float32, (B, 2 * D), "emb", temb.device)
    u = _output(u, torch.float32, (B, D), "u", temb.device)
    _check("adaln_f32_proj_fwd", L.adaln_f32_proj_fwd(_ptr(temb), _ptr(W), _ptr(bias), _ptr(emb), _ptr(u), B, D,
                                                      _stream(stream)))
    return emb, u


def adaln_f32_out_fwd(x, emb, out=None, mean=None, rstd=None, eps=1e-6, stream=None):
    """fp32 LayerNorm + modulation: (out [B,S,D], mean, rstd [B,S]), fp32."""
    L = load()
    B, S, D = x.shape
    x = _input(x, torch.float32, (B, S, D), "x")
    emb = _input(emb, torch.float32, (B, 2 * D), "emb")
    out = _output(out, torch.float32, (B, S, D), "out", x.device)
    mean = _output(mean, torch.float32, (B, S), "mean", x.device)
    rstd = _output(rstd, torch.float32, (B, S), "rstd", x.device)
    _check("adaln_f32_out_fwd", L.adaln_f32_out_fwd(_ptr(x), _ptr(emb), _ptr(out), _ptr(mean), _ptr(rstd), B, S, D,
                                                    float(eps), _stream(stream)))
    return out, mean, rstd


def adaln_f32_out_bwd(dy, x, emb, mean, rstd, dx=None, d_emb=None, workspace=None, stream=None):
    """fp32 backward of adaln_f32_out_fwd: (dx [B,S,D], d_emb [B,2D]), fp32."""
    L = load()
    B, S, D = x.shape
    dy = _input(dy, torch.float32, (B, S, D), "dy")
    x = _input(x, torch.float32, (B, S, D), "x")
    emb = _input(emb, torch.float32, (B, 2 * D), "emb")
    mean = _input(mean, torch.float32, (B, S), "mean")
    rstd = _input(rstd, torch.float32, (B, S), "rstd")
    dx = _output(dx, torch.float32, (B, S, D), "dx", x.device)
    d_emb = _output(d_emb, torch.float32, (B, 2 * D), "d_emb", x.device)
    ws, nws = _workspace(workspace, L.adaln_f32_out_bwd_workspace_bytes(B, S, D), x.device)
    _check("adaln_f32_out_bwd", L.adaln_f32_out_bwd(_ptr(dy), _ptr(x), _ptr(emb), _ptr(mean), _ptr(rstd), _ptr(dx),
                                                    _ptr(d_emb), _ptr(ws), nws, B, S, D, _stream(stream)))
    return dx, d_emb


def adaln_f32_out_bwd_workspace_bytes(B, S, D):
    return load().adaln_f32_out_bwd_workspace_bytes(B, S, D)


def adaln_f32_proj_bwd_workspace_bytes(B, D):
    return load().adaln_f32_proj_bwd_workspace_bytes(B, D)


def adaln_f32_proj_bwd(d_emb, temb, u, W, d_temb=None, dW_acc=None, db_acc=None, accumulate=False, want_w=True,
                       workspace=None, stream=None):
    """fp32 projection backward: (d_temb, dW_acc, db_acc); the accumulators are
    allocated here when not given and want_w."""
    L = load()
    B, D = temb.shape
    d_emb = _input(d_emb, torch.float32, (B, 2 * D), "d_emb")
    temb = _input(temb, torch.float32, (B, D), "temb")
    u = _input(u, torch.float32, (B, D), "u")
    W = _input(W, torch.float32, (2 * D, D), "W")
    d_temb = _output(d_temb, torch.float32, (B, D), "d_temb", temb.device)
    if want_w:
        dW_acc = _output(dW_acc, torch.float32, (2 * D, D), "dW_acc", temb.device)
        db_acc = _output(db_acc, torch.float32, (2 * D,), "db_acc", temb.device)
    ws, nws = _workspace(workspace, L.adaln_f32_proj_bwd_workspace_bytes(B, D), temb.device)
    _check("adaln_f32_proj_bwd", L.adaln_f32_proj_bwd(_ptr(d_emb), _ptr(temb), _ptr(u), _ptr(W), _ptr(d_temb),
                                                      _ptr(dW_acc), _ptr(db_acc), int(bool(accumulate)), _ptr(ws),
                                                      nws, B, D, _stream(stream)))
    return d_temb, dW_acc, db_acc


def adaln_scale_residual_norm_fwd(x, residual, gate, emb, r=None, out=None, mean=None, rstd=None, eps=1e-6,
                                  stream=None):
    """ScaleResidualLayerNormScaleShift forward: r = bf16(residual + bf16(gate
    * x)), then the LayerNorm + modulation of r.  Returns (r, out, mean, rstd)."""
    L = load()
    B, S, D = x.shape
    x = _input(x, torch.bfloat16, (B, S, D), "x")
    residual = _input(residual, torch.bfloat16, (B, S, D), "residual")
    gate = _input(gate, torch.bfloat16, (B, D), "gate")
    emb = _input(emb, torch.bfloat16, (B, 2 * D), "emb")
    r = _output(r, torch.bfloat16, (B, S, D), "r", x.device)
    out = _output(out, torch.bfloat16, (B, S, D), "out", x.device)
    mean = _output(mean, torch.float32, (B, S), "mean", x.device)
    rstd = _output(rstd, torch.float32, (B, S), "rstd", x.device)
    _check("adaln_scale_residual_norm_fwd",
           L.adaln_scale_residual_norm_fwd(_ptr(x), _ptr(residual), _ptr(gate), _ptr(emb), _ptr(r), _ptr(out),
                                           _ptr(mean), _ptr(rstd), B, S, D, float(eps), _stream(stream)))
    return r, out, mean, rstd


def adaln_scale_residual_norm_bwd_workspace_bytes(B, S, D):
    return load().adaln_scale_residual_norm_bwd_workspace_bytes(B, S, D)


def adaln_scale_residual_norm_bwd(d_out, d_r, x, r, gate, emb, mean, rstd, d_x=None, d_residual=None, d_emb=None,
                                  d_gate=None, workspace=None, stream=None):
    """Backward of adaln_scale_residual_norm_fwd; d_r (the gradient of r from
    its later uses) may be None.  Returns (d_x, d_residual, d_emb, d_gate)."""
    L = load()
    B, S, D = x.shape
    d_out = _input(d_out, torch.bfloat16, (B, S, D), "d_out")
    d_r = None if d_r is None else _input(d_r, torch.bfloat16, (B, S, D), "d_r")
    x = _input(x, torch.bfloat16, (B, S, D), "x")
    r = _input(r, torch.bfloat16, (B, S, D), "r")
    gate = _input(gate, torch.bfloat16, (B, D), "gate")
    emb = _input(emb, torch.bfloat16, (B, 2 * D), "emb")
    mean = _input(mean, torch.float32, (B, S), "mean")
    rstd = _input(rstd, torch.float32, (B, S), "rstd")
    d_x = _output(d_x, torch.bfloat16, (B, S, D), "d_x", x.device)
    d_residual = _output(d_residual, torch.bfloat16, (B, S, D), "d_residual", x.device)
    d_emb = _output(d_emb, torch.float32, (B, 2 * D), "d_emb", x.device)
    d_gate = _output(d_gate, torch.float32, (B, D), "d_gate", x.device)
    ws, nws = _workspace(workspace, L.adaln_scale_residual_norm_bwd_workspace_bytes(B, S, D), x.device)
    _check("adaln_scale_residual_norm_bwd",
           L.adaln_scale_residual_norm_bwd(_ptr(d_out), _ptr(d_r), _ptr(x), _ptr(r), _ptr(gate), _ptr(emb),
                                           _ptr(mean), _ptr(rstd), _ptr(d_x), _ptr(d_residual), _ptr(d_emb),
                                           _ptr(d_gate), _ptr(ws), nws, B, S, D, _stream(stream)))
    return d_x, d_residual, d_emb, d_gate


def adaln_out_bwd_noalloc(dy, x, emb, mean, rstd, dx=None, d_emb=None, stream=None):
    """adaln_out_bwd without a workspace, for callers that cannot allocate
    device memory at this point: the tree partials use a 24 MiB array inside
    the library.  dx and d_emb must be passed in for a call that allocates
    nothing (otherwise they are allocated here).  Returns (dx, d_emb)."""
    L = load()
    B, S, D = x.shape
    dy = _input(dy, torch.bfloat16, (B, S, D), "dy")
    x = _input(x, torch.bfloat16, (B, S, D), "x")
    emb = _input(emb, torch.bfloat16, (B, 2 * D), "emb")
    mean = _input(mean, torch.float32, (B, S), "mean")
    rstd = _input(rstd, torch.float32, (B, S), "rstd")
    dx = _output(dx, torch.bfloat16, (B, S, D), "dx", x.device)
    d_emb = _output(d_emb, torch.float32, (B, 2 * D), "d_emb", x.device)
    _check("adaln_out_bwd_noalloc", L.adaln_out_bwd_noalloc(_ptr(dy), _ptr(x), _ptr(emb), _ptr(mean), _ptr(rstd),
                                                            _ptr(dx), _ptr(d_emb), B, S, D, _stream(stream)))
    return dx, d_emb


def token_sum_tree_workspace_bytes(B, S, H):
    return load().token_sum_tree_workspace_bytes(B, S, H)


def token_sum_tree(inp, out=None, workspace=None, stream=None):
    """out[b,h] = the fixed 32-way Neumaier tree sum over s of inp[b,s,h] (fp32)."""
    L = load()
    B, S, H = inp.shape
    inp = _input(inp, torch.float32, (B, S, H), "in")
    out = _output(out, torch.float32, (B, H), "out", inp.device)
    ws, nws = _workspace(workspace, L.token_sum_tree_workspace_bytes(B, S, H), inp.device)
    _check("token_sum_tree", L.token_sum_tree(_ptr(inp), _ptr(out), B, S, H, _ptr(ws), nws, _stream(stream)))
    return out


def adaln_proj_bwd_workspace_bytes(B, D):
    return load().adaln_proj_bwd_workspace_bytes(B, D)


def adaln_proj_bwd(d_emb, temb, u, W, d_temb=None, dW_acc=None, db_acc=None, dW=None, db=None,
                   accumulate=False, workspace=None, stream=None):
    """Backward of adaln_proj_fwd.  Pass the gradient buffers you want (any of
    dW_acc/db_acc fp32 accumulators, dW/db bf16 outputs); returns
    (d_temb, dW_acc, db_acc, dW, db) with None for those not computed."""
    L = load()
    B, D = temb.shape
    d_emb = _input(d_emb, torch.float32, (B, 2 * D), "d_emb")
    temb = _input(temb, torch.bfloat16, (B, D), "temb")
    u = _input(u, torch.bfloat16, (B, D), "u")
    W = _input(W, torch.bfloat16, (2 * D, D), "W")
    dev = temb.device
    d_temb = _output(d_temb, torch.bfloat16, (B, D), "d_temb", dev)
    if dW_acc is not None:
        dW_acc = _output(dW_acc, torch.float32, (2 * D, D), "dW_acc", dev)
    if db_acc is not None:
        db_acc = _output(db_acc, torch.float32, (2 * D,), "db_acc", dev)
    if dW is not None:
        dW = _output(dW, torch.bfloat16, (2 * D, D), "dW", dev)
    if db is not None:
        db = _output(db, torch.bfloat16, (2 * D,), "db", dev)
    ws, nws = _workspace(workspace, L.adaln_proj_bwd_workspace_bytes(B, D), dev)
    _check("adaln_proj_bwd", L.adaln_proj_bwd(_ptr(d_emb), _ptr(temb), _ptr(u), _ptr(W), _ptr(d_temb),
                                              _ptr(dW_acc), _ptr(db_acc), _ptr(dW), _ptr(db), int(bool(accumulate)),
                                              _ptr(ws), nws, B, D, _stream(stream)))
    return d_temb, dW_acc, db_acc, dW, db


def adaln_proj_wgrad_rows(d_emb, u, n0, n1, dW_acc=None, db_acc=None, dW=None, db=None, accumulate=False,
                          stream=None):
    """dW/db of the output rows n0 <= n < n1 over all given samples (ascending);
    pass the row-block buffers you want ([n1-n0, D] and [n1-n0]).  Returns
    (dW_acc, db_acc, dW, db) with None for those not computed."""
    L = load()
    B, D = u.shape
    d_emb = _input(d_emb, torch.float32, (B, 2 * D), "d_emb")
    u = _input(u, torch.bfloat16, (B, D), "u")
    R = n1 - n0
    dev = u.device
    if dW_acc is not None:
        dW_acc = _output(dW_acc, torch.float32, (R, D), "dW_acc", dev)
    if db_acc is not None:
        db_acc = _output(db_acc, torch.float32, (R,), "db_acc", dev)
    if dW is not None:
        dW = _output(dW, torch.bfloat16, (R, D), "dW", dev)
    if db is not None:
        db = _output(db, torch.bfloat16, (R,), "db", dev)
    _check("adaln_proj_wgrad_rows", L.adaln_proj_wgrad_rows(_ptr(d_emb), _ptr(u), int(n0), int(n1), _ptr(dW_acc),
                                                            _ptr(db_acc), _ptr(dW), _ptr(db), int(bool(accumulate)),
                                                            B, D, _stream(stream)))
    return dW_acc, db_acc, dW, db
