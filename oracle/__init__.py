"""CPU oracle for the AdaLN ``norm_out`` operator (test infrastructure).

The arithmetic lives in ``adaln_oracle.c`` (plain C, fp64 with the operator's
rounding points, IEEE as written, no FMA contraction).  This module only
compiles it with gcc and marshals numpy arrays into it.

Only the tests, the smoke check and the benchmark's CPU-baseline leg use this
package; the CUDA library never imports it, and it imports nothing from the
CUDA library.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "adaln_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``liboracle.so`` next to its source."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I = ctypes.c_int
        F = ctypes.c_float
        Dd = ctypes.c_double
        Lg = ctypes.c_long
        sig = {
            "oracle_silu_bf16": [P, P, Lg],
            "oracle_dsilu_f64": [P, P, Lg],
            "oracle_proj_fwd": [P, P, P, P, I, I],
            "oracle_proj_fwd_rows": [P, P, P, P, I, I, I, I],
            "oracle_proj_bwd_rows": [P, P, P, P, P, P, I, I, I, I],
            "oracle_proj_fwd_f64": [P, P, P, P, I, I],
            "oracle_out_fwd": [P, P, F, P, P, P, I, I, I],
            "oracle_out_fwd_f64": [P, P, P, Dd, P, I, I, I],
            "oracle_out_bwd": [P, P, P, F, P, P, I, I, I],
            "oracle_out_bwd_f64": [P, P, P, Dd, P, P, P, I, I, I],
            "oracle_token_sum_f64": [P, P, I, I, I],
            "oracle_token_tree_f32": [P, P, I, I, I],
            "oracle_bwd_products_f32": [P, P, P, P, P, I, I, I],
            "oracle_proj_bwd": [P, P, P, P, P, P, I, I],
            "oracle_proj_bwd_f64": [P, P, P, P, P, P, I, I],
            "oracle_wgrad_seq_f32": [P, P, P, P, I, I, I],
            "oracle_wgrad_seq_f32_rows": [P, P, P, I, P, P, I, I],
            "oracle_bf16_from_f64": [P, P, Lg],
            "oracle_res_fwd": [P, P, P, P, F, P, P, P, P, I, I, I],
            "oracle_res_bwd_tail": [P, P, P, P, P, P, P, I, I, I],
            "oracle_res_bwd": [P, P, P, P, P, P, F, P, P, P, P, I, I, I],
            "oracle_res_gate_products_f32": [P, P, P, Lg],
            "oracle_f32_proj_fwd": [P, P, P, P, P, I, I],
            "oracle_f32_out_fwd": [P, P, F, P, P, P, I, I, I],
            "oracle_f32_out_bwd": [P, P, P, F, P, P, I, I, I],
            "oracle_f32_bwd_products": [P, P, P, P, P, I, I, I],
            "oracle_f32_proj_bwd": [P, P, P, P, P, P, I, I],
            "oracle_f32_wgrad_seq": [P, P, P, P, I, I, I],
            "oracle_proj_out": [P, P, P, P, Lg, I, I],
        }
        for name, args in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = None
        _lib = L
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


EPS = np.float32(1e-6)


# --- projection -----------------------------------------------------------

def silu_bf16(t):
    t = _c(t, np.uint16)
    u = np.empty_like(t)
    _load().oracle_silu_bf16(_p(t), _p(u), t.size)
    return u


def dsilu_f64(t):
    t = _c(t, np.float64)
    o = np.empty_like(t)
    _load().oracle_dsilu_f64(_p(t), _p(o), t.size)
    return o


def proj_fwd(temb, W, b):
    """emb[B, 2D] (bf16 bits) = bf16(bf16(silu(temb)) @ W^T + b)."""
    temb, W, b = _c(temb, np.uint16), _c(W, np.uint16), _c(b, np.uint16)
    B, D = temb.shape
    assert W.shape == (2 * D, D) and b.shape == (2 * D,)
    emb = np.empty((B, 2 * D), dtype=np.uint16)
    _load().oracle_proj_fwd(_p(temb), _p(W), _p(b), _p(emb), B, D)
    return emb


def proj_fwd_rows(temb, W, b, n0, n1, emb=None):
    """The projection for the output rows n0 <= n < n1 only (others of
    ``emb`` are left as given)."""
    temb, W, b = _c(temb, np.uint16), _c(W, np.uint16), _c(b, np.uint16)
    B, D = temb.shape
    assert 0 <= n0 <= n1 <= 2 * D
    emb = np.zeros((B, 2 * D), dtype=np.uint16) if emb is None else _c(emb, np.uint16)
    _load().oracle_proj_fwd_rows(_p(temb), _p(W), _p(b), _p(emb), B, D, n0, n1)
    return emb


def proj_fwd_f64(temb, W, b):
    temb, W, b = _c(temb, np.float64), _c(W, np.float64), _c(b, np.float64)
    B, D = temb.shape
    emb = np.empty((B, 2 * D), dtype=np.float64)
    _load().oracle_proj_fwd_f64(_p(temb), _p(W), _p(b), _p(emb), B, D)
    return emb


# --- LayerNorm + modulation -------------------------------------------------

def out_fwd(x, emb, eps=EPS):
    """(out bf16 bits [B,S,D], mean fp32 [B,S], rstd fp32 [B,S])."""
    x, emb = _c(x, np.uint16), _c(emb, np.uint16)
    B, S, D = x.shape
    assert emb.shape == (B, 2 * D)
    out = np.empty_like(x)
    mean = np.empty((B, S), dtype=np.float32)
    rstd = np.empty((B, S), dtype=np.float32)
    _load().oracle_out_fwd(_p(x), _p(emb), float(eps), _p(out), _p(mean), _p(rstd), B, S, D)
    return out, mean, rstd


def out_fwd_f64(x, scale, shift, eps=1e-6):
    x, scale, shift = _c(x, np.float64), _c(scale, np.float64), _c(shift, np.float64)
    B, S, D = x.shape
    out = np.empty_like(x)
    _load().oracle_out_fwd_f64(_p(x), _p(scale), _p(shift), float(eps), _p(out), B, S, D)
    return out


def out_bwd(dy, x, emb, eps=EPS):
    """(dx bf16 bits [B,S,D], d_emb fp32 [B,2D] = [d_scale | d_shift])."""
    dy, x, emb = _c(dy, np.uint16), _c(x, np.uint16), _c(emb, np.uint16)
    B, S, D = x.shape
    dx = np.empty_like(x)
    d_emb = np.empty((B, 2 * D), dtype=np.float32)
    _load().oracle_out_bwd(_p(dy), _p(x), _p(emb), float(eps), _p(dx), _p(d_emb), B, S, D)
    return dx, d_emb


def out_bwd_f64(dy, x, scale, eps=1e-6):
    dy, x, scale = _c(dy, np.float64), _c(x, np.float64), _c(scale, np.float64)
    B, S, D = x.shape
    dx = np.empty_like(x)
    ds = np.empty((B, D), dtype=np.float64)
    dh = np.empty((B, D), dtype=np.float64)
    _load().oracle_out_bwd_f64(_p(dy), _p(x), _p(scale), float(eps), _p(dx), _p(ds), _p(dh), B, S, D)
    return dx, ds, dh


# --- token sums -----------------------------------------------------------

def token_sum_f64(a):
    a = _c(a, np.float32)
    B, S, H = a.shape
    out = np.empty((B, H), dtype=np.float64)
    _load().oracle_token_sum_f64(_p(a), _p(out), B, S, H)
    return out


def token_tree_f32(a):
    a = _c(a, np.float32)
    B, S, H = a.shape
    assert S >= 1
    out = np.empty((B, H), dtype=np.float32)
    _load().oracle_token_tree_f32(_p(a), _p(out), B, S, H)
    return out


def bwd_products_f32(dy, x, mean, rstd):
    dy, x = _c(dy, np.uint16), _c(x, np.uint16)
    mean, rstd = _c(mean, np.float32), _c(rstd, np.float32)
    B, S, D = x.shape
    prod = np.empty((B, S, 2 * D), dtype=np.float32)
    _load().oracle_bwd_products_f32(_p(dy), _p(x), _p(mean), _p(rstd), _p(prod), B, S, D)
    return prod


# --- projection backward --------------------------------------------------

def proj_bwd(d_emb, temb, W, want_dW=True):
    """(d_temb bf16 bits [B,D], dW fp64 [2D,D] or None, db fp64 [2D])."""
    d_emb, temb, W = _c(d_emb, np.float32), _c(temb, np.uint16), _c(W, np.uint16)
    B, D = temb.shape
    d_temb = np.empty((B, D), dtype=np.uint16)
    dW = np.empty((2 * D, D), dtype=np.float64) if want_dW else None
    db = np.empty(2 * D, dtype=np.float64)
    _load().oracle_proj_bwd(_p(d_emb), _p(temb), _p(W), _p(d_temb), _p(dW), _p(db), B, D)
    return d_temb, dW, db


def proj_bwd_rows(d_emb, temb, W, n0, n1, want_dW=True):
    """The projection backward's sums over the output rows n0 <= n < n1:
    (d_silu partial fp64 [B,D], dW fp64 [2D,D] (rows n0..n1 filled) or None,
    db fp64 [2D] (rows n0..n1 filled))."""
    d_emb, temb, W = _c(d_emb, np.float32), _c(temb, np.uint16), _c(W, np.uint16)
    B, D = temb.shape
    assert 0 <= n0 <= n1 <= 2 * D
    d_silu = np.empty((B, D), dtype=np.float64)
    dW = np.zeros((2 * D, D), dtype=np.float64) if want_dW else None
    db = np.zeros(2 * D, dtype=np.float64)
    _load().oracle_proj_bwd_rows(_p(d_emb), _p(temb), _p(W), _p(d_silu), _p(dW), _p(db), B, D, n0, n1)
    return d_silu, dW, db


def proj_bwd_f64(d_emb, temb, W):
    d_emb, temb, W = _c(d_emb, np.float64), _c(temb, np.float64), _c(W, np.float64)
    B, D = temb.shape
    d_temb = np.empty((B, D), dtype=np.float64)
    dW = np.empty((2 * D, D), dtype=np.float64)
    db = np.empty(2 * D, dtype=np.float64)
    _load().oracle_proj_bwd_f64(_p(d_emb), _p(temb), _p(W), _p(d_temb), _p(dW), _p(db), B, D)
    return d_temb, dW, db


def wgrad_seq_f32(d_emb, temb, dW_acc=None, db_acc=None, accumulate=False):
    """(dW_acc fp32 [2D,D], db_acc fp32 [2D]) in the operator's sequential order."""
    d_emb, temb = _c(d_emb, np.float32), _c(temb, np.uint16)
    B, D = temb.shape
    dW = np.zeros((2 * D, D), np.float32) if dW_acc is None else np.array(dW_acc, dtype=np.float32, copy=True)
    db = np.zeros(2 * D, np.float32) if db_acc is None else np.array(db_acc, dtype=np.float32, copy=True)
    _load().oracle_wgrad_seq_f32(_p(d_emb), _p(temb), _p(dW), _p(db), int(bool(accumulate)), B, D)
    return dW, db


def wgrad_seq_f32_rows(d_emb, temb, rows):
    """Rows `rows` of (dW_acc, db_acc) of wgrad_seq_f32 started from +0:
    (dW fp32 [len(rows), D], db fp32 [len(rows)])."""
    d_emb, temb = _c(d_emb, np.float32), _c(temb, np.uint16)
    B, D = temb.shape
    rows = _c(rows, np.int32)
    assert rows.ndim == 1 and np.all((rows >= 0) & (rows < 2 * D))
    dW = np.empty((len(rows), D), np.float32)
    db = np.empty(len(rows), np.float32)
    _load().oracle_wgrad_seq_f32_rows(_p(d_emb), _p(temb), _p(rows), len(rows), _p(dW), _p(db), B, D)
    return dW, db


# --- block-level modulated norm with a gated residual ----------------------

def res_fwd(x, residual, gate, emb, eps=EPS):
    """(r, out, mean, rstd): r = bf16(residual + bf16(gate * x)), then the
    LayerNorm + modulation of r."""
    x, residual = _c(x, np.uint16), _c(residual, np.uint16)
    gate, emb = _c(gate, np.uint16), _c(emb, np.uint16)
    B, S, D = x.shape
    assert residual.shape == x.shape and gate.shape == (B, D) and emb.shape == (B, 2 * D)
    r = np.empty_like(x)
    out = np.empty_like(x)
    mean = np.empty((B, S), dtype=np.float32)
    rstd = np.empty((B, S), dtype=np.float32)
    _load().oracle_res_fwd(_p(x), _p(residual), _p(gate), _p(emb), float(eps), _p(r), _p(out), _p(mean),
                           _p(rstd), B, S, D)
    return r, out, mean, rstd


def res_bwd_tail(dr_ln, d_r, x, gate):
    """(d_x, d_residual, d_gate) from the LayerNorm input's gradient dr_ln
    (bf16) and the residual output's gradient d_r (bf16, or None)."""
    dr_ln, x, gate = _c(dr_ln, np.uint16), _c(x, np.uint16), _c(gate, np.uint16)
    B, S, D = x.shape
    dr = None if d_r is None else _c(d_r, np.uint16)
    d_x = np.empty_like(x)
    d_res = np.empty_like(x)
    d_gate = np.empty((B, D), dtype=np.float32)
    _load().oracle_res_bwd_tail(_p(dr_ln), None if dr is None else _p(dr), _p(x), _p(gate), _p(d_x), _p(d_res),
                                _p(d_gate), B, S, D)
    return d_x, d_res, d_gate


def res_bwd(d_out, d_r, x, r, gate, emb, eps=EPS):
    """(d_x, d_residual, d_emb, d_gate): the whole backward of res_fwd."""
    d_out, x, r = _c(d_out, np.uint16), _c(x, np.uint16), _c(r, np.uint16)
    gate, emb = _c(gate, np.uint16), _c(emb, np.uint16)
    B, S, D = x.shape
    dr = None if d_r is None else _c(d_r, np.uint16)
    d_x = np.empty_like(x)
    d_res = np.empty_like(x)
    d_emb = np.empty((B, 2 * D), dtype=np.float32)
    d_gate = np.empty((B, D), dtype=np.float32)
    _load().oracle_res_bwd(_p(d_out), None if dr is None else _p(dr), _p(x), _p(r), _p(gate), _p(emb), float(eps),
                           _p(d_x), _p(d_res), _p(d_emb), _p(d_gate), B, S, D)
    return d_x, d_res, d_emb, d_gate


def res_gate_products_f32(gr, x):
    """bf16(gr * x) as fp32: the token products of d_gate."""
    gr, x = _c(gr, np.uint16), _c(x, np.uint16)
    assert gr.shape == x.shape
    prod = np.empty(x.shape, dtype=np.float32)
    _load().oracle_res_gate_products_f32(_p(gr), _p(x), _p(prod), x.size)
    return prod


# --- proj_out ------------------------------------------------------------------

def proj_out(out, Wp, bp):
    """y [..., J] (bf16 bits) = bf16(out @ Wp^T + bp) for out [..., D] bf16 bits."""
    out, Wp, bp = _c(out, np.uint16), _c(Wp, np.uint16), _c(bp, np.uint16)
    J, D = Wp.shape
    assert out.shape[-1] == D and bp.shape == (J,)
    R = out.size // D
    y = np.empty(out.shape[:-1] + (J,), dtype=np.uint16)
    _load().oracle_proj_out(_p(out), _p(Wp), _p(bp), _p(y), R, D, J)
    return y


# --- fp32 execution dtype ----------------------------------------------------

def _f(a):
    return _c(a, np.float32)


def f32_proj_fwd(temb, W, b):
    """(emb [B,2D] fp32, u [B,D] fp32) of the fp32 operator."""
    temb, W, b = _f(temb), _f(W), _f(b)
    B, D = temb.shape
    emb = np.empty((B, 2 * D), np.float32)
    u = np.empty((B, D), np.float32)
    _load().oracle_f32_proj_fwd(_p(temb), _p(W), _p(b), _p(emb), _p(u), B, D)
    return emb, u


def f32_out_fwd(x, emb, eps=EPS):
    x, emb = _f(x), _f(emb)
    B, S, D = x.shape
    out = np.empty_like(x)
    mean = np.empty((B, S), np.float32)
    rstd = np.empty((B, S), np.float32)
    _load().oracle_f32_out_fwd(_p(x), _p(emb), float(eps), _p(out), _p(mean), _p(rstd), B, S, D)
    return out, mean, rstd


def f32_out_bwd(dy, x, emb, eps=EPS):
    dy, x, emb = _f(dy), _f(x), _f(emb)
    B, S, D = x.shape
    dx = np.empty_like(x)
    d_emb = np.empty((B, 2 * D), np.float32)
    _load().oracle_f32_out_bwd(_p(dy), _p(x), _p(emb), float(eps), _p(dx), _p(d_emb), B, S, D)
    return dx, d_emb


def f32_bwd_products(dy, x, mean, rstd):
    dy, x, mean, rstd = _f(dy), _f(x), _f(mean), _f(rstd)
    B, S, D = x.shape
    prod = np.empty((B, S, 2 * D), np.float32)
    _load().oracle_f32_bwd_products(_p(dy), _p(x), _p(mean), _p(rstd), _p(prod), B, S, D)
    return prod


def f32_proj_bwd(d_emb, temb, W, want_dW=True):
    d_emb, temb, W = _f(d_emb), _f(temb), _f(W)
    B, D = temb.shape
    d_temb = np.empty((B, D), np.float32)
    dW = np.empty((2 * D, D), np.float32) if want_dW else None
    db = np.empty(2 * D, np.float32) if want_dW else None
    _load().oracle_f32_proj_bwd(_p(d_emb), _p(temb), _p(W), _p(d_temb), _p(dW), _p(db), B, D)
    return d_temb, dW, db


def f32_wgrad_seq(d_emb, u, dW_acc=None, db_acc=None, accumulate=False):
    d_emb, u = _f(d_emb), _f(u)
    B, D = u.shape
    dW = np.zeros((2 * D, D), np.float32) if dW_acc is None else _f(dW_acc).copy()
    db = np.zeros(2 * D, np.float32) if db_acc is None else _f(db_acc).copy()
    _load().oracle_f32_wgrad_seq(_p(d_emb), _p(u), _p(dW), _p(db), int(bool(accumulate)), B, D)
    return dW, db


def bf16_from_f64(a):
    a = _c(a, np.float64)
    h = np.empty(a.shape, dtype=np.uint16)
    _load().oracle_bf16_from_f64(_p(a), _p(h), a.size)
    return h
