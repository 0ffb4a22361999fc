"""The C ABI on the host: the library loads, exports every function the
header declares, and rejects each invalid argument with its status before
anything is launched.

The pointers here are fake addresses that are never dereferenced: every call
below fails one of the host checks, which run before the device check and
before any launch.  The single call with all arguments valid runs only on a
machine without a GPU, where it must stop at the device check.
"""

from __future__ import annotations

import ctypes

import pytest
import torch

from invariant_dit_adaln_gb300 import binding, build

OK, NULL, SHAPE, ALIGN, ALIAS, WORKSPACE, DEVICE, CUDA, ARG = range(9)
TB = 1 << 40  # fake buffers sit 1 TiB apart, so they never overlap


@pytest.fixture(scope="module")
def L():
    build.build()
    return binding.load()


@pytest.fixture
def no_gpu():
    """Calls with fake pointers run only where no GPU is visible: should a
    case pass every host check by mistake, it must not reach a launch."""
    if torch.cuda.is_available():
        pytest.skip("fake-pointer checks run only on machines without a GPU")


def fake(i, off=0):
    return ctypes.c_void_p((i + 1) * TB + off)


def test_library_exports_every_declared_symbol(L):
    names = binding.declared_symbols()
    assert len(names) == 23, names
    for n in names:
        assert hasattr(L, n), n
    assert L.adaln_version() >> 16 == 1


def test_status_strings(L):
    for s in range(9):
        assert binding.status_string(s).startswith("ADALN_")
    assert "unknown" in binding.status_string(99)


def test_workspace_sizes(L):
    D = 3072
    # tree partials (sum, correction) per 32-token tile
    assert L.adaln_out_bwd_workspace_bytes(2, 4096, D) == 2 * 2 * 128 * 6144 * 4
    assert L.adaln_out_bwd_workspace_bytes(2, 33, D) == 2 * 2 * 2 * 6144 * 4
    assert L.adaln_out_bwd_workspace_bytes(0, 33, D) == 0
    assert L.adaln_out_bwd_workspace_bytes(2, 0, D) == 0
    assert L.token_sum_tree_workspace_bytes(1, 1, 4) == 256  # 32 bytes, rounded to 256
    assert L.adaln_proj_bwd_workspace_bytes(2, D) == 24 * 2 * 3072 * 4  # ceil(2D / 256) slabs
    assert L.adaln_proj_bwd_workspace_bytes(0, D) == 0


# --- adaln_proj_fwd ---------------------------------------------------------

def proj_fwd(L, temb=0, W=1, b=2, emb=3, u=4, B=2, D=3072):
    p = [None if a is None else (fake(a) if isinstance(a, int) else a) for a in (temb, W, b, emb, u)]
    return L.adaln_proj_fwd(*p, B, D, None)


def test_proj_fwd_checks(L, no_gpu):
    assert proj_fwd(L, temb=None) == NULL
    assert proj_fwd(L, u=None) == NULL
    assert proj_fwd(L, D=12) == SHAPE
    assert proj_fwd(L, D=0) == SHAPE
    assert proj_fwd(L, D=8200) == SHAPE
    assert proj_fwd(L, B=-1) == SHAPE
    assert proj_fwd(L, W=fake(1, 8)) == ALIGN
    assert proj_fwd(L, emb=fake(3, 2)) == ALIGN
    assert proj_fwd(L, emb=fake(1, 4096)) == ALIAS      # emb inside W
    assert proj_fwd(L, u=fake(3, 16)) == ALIAS          # u overlaps emb
    assert proj_fwd(L, u=fake(0)) == ALIAS              # u is temb


# --- adaln_out_fwd ----------------------------------------------------------

def out_fwd(L, x=0, emb=1, out=2, mean=3, rstd=4, B=2, S=33, D=3072, eps=1e-6):
    p = [None if a is None else (fake(a) if isinstance(a, int) else a) for a in (x, emb, out, mean, rstd)]
    return L.adaln_out_fwd(*p, B, S, D, eps, None)


def test_out_fwd_checks(L, no_gpu):
    assert out_fwd(L, mean=None) == NULL
    assert out_fwd(L, S=-1) == SHAPE
    assert out_fwd(L, S=262145) == SHAPE
    assert out_fwd(L, B=65536) == SHAPE
    assert out_fwd(L, D=4) == SHAPE
    assert out_fwd(L, eps=float("nan")) == ARG
    assert out_fwd(L, eps=-1.0) == ARG
    assert out_fwd(L, x=fake(0, 2)) == ALIGN
    assert out_fwd(L, rstd=fake(4, 4)) == ALIGN
    assert out_fwd(L, out=fake(0, 1024)) == ALIAS        # out inside x
    assert out_fwd(L, rstd=fake(3, 16)) == ALIAS         # rstd overlaps mean
    # mean placed right after out: no overlap -> passes the alias check (fails later)
    assert out_fwd(L, mean=fake(2, 2 * 33 * 3072 * 2), rstd=fake(2, 2 * 33 * 3072 * 2 + 1024), S=33) != ALIAS


# --- adaln_out_bwd ----------------------------------------------------------

def out_bwd(L, dy=0, x=1, emb=2, mean=3, rstd=4, dx=5, d_emb=6, ws=7, nws=None, B=2, S=33, D=3072):
    p = [None if a is None else (fake(a) if isinstance(a, int) else a) for a in (dy, x, emb, mean, rstd, dx, d_emb, ws)]
    if nws is None:
        nws = L.adaln_out_bwd_workspace_bytes(B, S, D)
    return L.adaln_out_bwd(*p, nws, B, S, D, None)


def test_out_bwd_checks(L, no_gpu):
    assert out_bwd(L, dy=None) == NULL
    assert out_bwd(L, d_emb=None) == NULL
    assert out_bwd(L, D=3004) == SHAPE
    assert out_bwd(L, S=1 << 20) == SHAPE
    assert out_bwd(L, ws=fake(7, 8)) == ALIGN
    assert out_bwd(L, mean=fake(3, 4)) == ALIGN
    assert out_bwd(L, dx=fake(1)) == ALIAS               # dx is x
    assert out_bwd(L, d_emb=fake(2, 16)) == ALIAS        # d_emb inside emb
    assert out_bwd(L, ws=fake(5, 4096)) == ALIAS         # workspace inside dx
    assert out_bwd(L, nws=100) == WORKSPACE
    assert out_bwd(L, ws=None) == WORKSPACE
    assert out_bwd(L, nws=L.adaln_out_bwd_workspace_bytes(2, 33, 3072) - 1) == WORKSPACE


def out_bwd_noalloc(L, dy=0, x=1, emb=2, mean=3, rstd=4, dx=5, d_emb=6, B=2, S=33, D=3072):
    p = [None if a is None else (fake(a) if isinstance(a, int) else a) for a in (dy, x, emb, mean, rstd, dx, d_emb)]
    return L.adaln_out_bwd_noalloc(*p, B, S, D, None)


def test_out_bwd_noalloc_checks(L, no_gpu):
    """The checks of adaln_out_bwd in the same order, the array's size limit
    counted with the sizes; the device is checked before the library's array
    is looked up."""
    assert out_bwd_noalloc(L, D=3004) == SHAPE
    assert out_bwd_noalloc(L, S=8192 + 32) == SHAPE       # partials beyond the 24 MiB array
    assert out_bwd_noalloc(L, dy=None, S=8192 + 32) == SHAPE
    assert out_bwd_noalloc(L, dy=None) == NULL
    assert out_bwd_noalloc(L, mean=fake(3, 4)) == ALIGN
    assert out_bwd_noalloc(L, dx=fake(1)) == ALIAS
    assert out_bwd_noalloc(L) == DEVICE                     # valid arguments: the device check comes next


# --- token_sum_tree ---------------------------------------------------------

def tree(L, inp=0, out=1, ws=2, nws=None, B=2, S=33, H=6144):
    p = [None if a is None else (fake(a) if isinstance(a, int) else a) for a in (inp, out, ws)]
    if nws is None:
        nws = L.token_sum_tree_workspace_bytes(B, S, H)
    return L.token_sum_tree(p[0], p[1], B, S, H, p[2], nws, None)


def test_token_sum_tree_checks(L, no_gpu):
    assert tree(L, inp=None) == NULL
    assert tree(L, H=6) == SHAPE
    assert tree(L, H=0) == SHAPE
    assert tree(L, S=-3) == SHAPE
    assert tree(L, out=fake(1, 4)) == ALIGN
    assert tree(L, out=fake(0, 64)) == ALIAS
    assert tree(L, ws=fake(1, 1024)) == ALIAS
    assert tree(L, nws=16) == WORKSPACE


# --- adaln_proj_bwd ---------------------------------------------------------

def proj_bwd(L, d_emb=0, temb=1, u=2, W=3, d_temb=4, dW_acc=5, db_acc=6, dW=7, db=8, acc=0, ws=9, nws=None,
             B=2, D=3072):
    p = [None if a is None else (fake(a) if isinstance(a, int) else a)
         for a in (d_emb, temb, u, W, d_temb, dW_acc, db_acc, dW, db)]
    wsp = None if ws is None else (fake(ws) if isinstance(ws, int) else ws)
    if nws is None:
        nws = L.adaln_proj_bwd_workspace_bytes(B, D)
    return L.adaln_proj_bwd(*p, acc, wsp, nws, B, D, None)


def test_proj_bwd_checks(L, no_gpu):
    assert proj_bwd(L, u=None) == NULL
    assert proj_bwd(L, d_temb=None) == NULL
    assert proj_bwd(L, D=7) == SHAPE
    assert proj_bwd(L, acc=2) == ARG
    assert proj_bwd(L, acc=1, dW_acc=None) == ARG        # accumulate needs the fp32 accumulator
    assert proj_bwd(L, acc=1, db_acc=None) == ARG
    assert proj_bwd(L, dW=fake(7, 2)) == ALIGN
    assert proj_bwd(L, dW=fake(3, 64)) == ALIAS          # dW inside W
    assert proj_bwd(L, dW_acc=fake(0)) == ALIAS          # accumulator is d_emb
    assert proj_bwd(L, db=fake(6, 16)) == ALIAS          # db inside db_acc
    assert proj_bwd(L, nws=8) == WORKSPACE
    assert proj_bwd(L, ws=None) == WORKSPACE


def wgrad_rows(L, d_emb=0, u=1, n0=0, n1=100, dW_acc=2, db_acc=3, dW=4, db=5, acc=0, B=2, D=3072):
    p = [None if a is None else (fake(a) if isinstance(a, int) else a) for a in (d_emb, u, dW_acc, db_acc, dW, db)]
    return L.adaln_proj_wgrad_rows(p[0], p[1], n0, n1, p[2], p[3], p[4], p[5], acc, B, D, None)


def test_proj_wgrad_rows_checks(L, no_gpu):
    assert wgrad_rows(L, n1=6145) == SHAPE                 # beyond 2D rows
    assert wgrad_rows(L, n0=10, n1=5) == SHAPE
    assert wgrad_rows(L, n0=-1) == SHAPE
    assert wgrad_rows(L, acc=3) == ARG
    assert wgrad_rows(L, acc=1, dW_acc=None) == ARG
    assert wgrad_rows(L, u=None) == NULL
    assert wgrad_rows(L, dW=fake(4, 8)) == ALIGN
    assert wgrad_rows(L, dW=fake(0, 64)) == ALIAS            # dW inside d_emb
    assert wgrad_rows(L) == DEVICE                          # valid: the device check comes next


# --- adaln_scale_residual_norm_fwd / _bwd ------------------------------------

def res_fwd(L, x=0, residual=1, gate=2, emb=3, r=4, out=5, mean=6, rstd=7, B=2, S=33, D=3072, eps=1e-6):
    p = [None if a is None else (fake(a) if isinstance(a, int) else a)
         for a in (x, residual, gate, emb, r, out, mean, rstd)]
    return L.adaln_scale_residual_norm_fwd(*p, B, S, D, ctypes.c_float(eps), None)


def res_bwd(L, d_out=0, d_r=1, x=2, r=3, gate=4, emb=5, mean=6, rstd=7, d_x=8, d_res=9, d_emb=10, d_gate=11,
            ws=12, nws=None, B=2, S=33, D=3072):
    p = [None if a is None else (fake(a) if isinstance(a, int) else a)
         for a in (d_out, d_r, x, r, gate, emb, mean, rstd, d_x, d_res, d_emb, d_gate)]
    wsp = None if ws is None else (fake(ws) if isinstance(ws, int) else ws)
    if nws is None:
        nws = L.adaln_scale_residual_norm_bwd_workspace_bytes(B, S, D)
    return L.adaln_scale_residual_norm_bwd(*p, wsp, nws, B, S, D, None)


def test_scale_residual_norm_checks(L, no_gpu):
    assert L.adaln_scale_residual_norm_bwd_workspace_bytes(2, 33, 3072) == L.adaln_out_bwd_workspace_bytes(2, 33, 3072)
    assert res_fwd(L, D=12) == SHAPE
    assert res_fwd(L, eps=-1.0) == ARG
    assert res_fwd(L, gate=None) == NULL
    assert res_fwd(L, r=None) == NULL
    assert res_fwd(L, r=fake(4, 8)) == ALIGN
    assert res_fwd(L, r=fake(1, 64)) == ALIAS             # r inside residual (no in-place form)
    assert res_fwd(L, out=fake(4, 1024)) == ALIAS         # out overlaps r
    assert res_fwd(L) == DEVICE
    assert res_bwd(L, S=-1) == SHAPE
    assert res_bwd(L, x=None) == NULL
    assert res_bwd(L, d_gate=None) == NULL
    assert res_bwd(L, d_r=None) == DEVICE                 # d_r is optional
    assert res_bwd(L, d_x=fake(8, 2)) == ALIGN
    assert res_bwd(L, d_res=fake(1, 0)) == ALIAS          # d_residual is d_r
    assert res_bwd(L, d_gate=fake(12, 0)) == ALIAS        # d_gate inside the workspace
    assert res_bwd(L, nws=16) == WORKSPACE
    assert res_bwd(L) == DEVICE


# --- adaln_out_fwd_proj --------------------------------------------------------

def test_out_fwd_proj_checks(L, no_gpu):
    F = ctypes.c_float

    def call(x=0, emb=1, Wp=2, bp=3, out=4, mean=5, rstd=6, y=7, B=2, S=33, D=3072, J=64, eps=1e-6):
        p = [None if a is None else (fake(a) if isinstance(a, int) else a) for a in (x, emb, Wp, bp, out, mean, rstd, y)]
        return L.adaln_out_fwd_proj(*p, B, S, D, J, F(eps), None)

    assert call(J=32) == SHAPE
    assert call(D=3080) == SHAPE           # not a multiple of 64
    assert call(B=65535, S=262144) == SHAPE
    assert call(eps=float("nan")) == ARG
    assert call(Wp=None) == NULL
    assert call(y=fake(7, 2)) == ALIGN
    assert call(y=fake(4, 1024)) == ALIAS  # y inside out
    assert call() == DEVICE


# --- fp32 execution dtype ------------------------------------------------------

def test_f32_checks(L, no_gpu):
    F = ctypes.c_float
    # projection forward: D <= 4096
    assert L.adaln_f32_proj_fwd(fake(0), fake(1), fake(2), fake(3), fake(4), 2, 8192, None) == SHAPE
    assert L.adaln_f32_proj_fwd(fake(0), None, fake(2), fake(3), fake(4), 2, 3072, None) == NULL
    assert L.adaln_f32_proj_fwd(fake(0), fake(1), fake(2), fake(3, 4), fake(4), 2, 3072, None) == ALIGN
    assert L.adaln_f32_proj_fwd(fake(0), fake(1), fake(2), fake(1, 64), fake(4), 2, 3072, None) == ALIAS
    assert L.adaln_f32_proj_fwd(fake(0), fake(1), fake(2), fake(3), fake(4), 2, 3072, None) == DEVICE
    # LayerNorm forward
    assert L.adaln_f32_out_fwd(fake(0), fake(1), fake(2), fake(3), fake(4), 2, 33, 4104, F(1e-6), None) == SHAPE
    assert L.adaln_f32_out_fwd(fake(0), fake(1), fake(2), fake(3), fake(4), 2, 33, 3072, F(-1.0), None) == ARG
    assert L.adaln_f32_out_fwd(fake(0), fake(1), fake(0, 16), fake(3), fake(4), 2, 33, 3072, F(1e-6), None) == ALIAS
    assert L.adaln_f32_out_fwd(fake(0), fake(1), fake(2), fake(3), fake(4), 2, 33, 3072, F(1e-6), None) == DEVICE
    # backward
    nws = L.adaln_f32_out_bwd_workspace_bytes(2, 33, 3072)
    assert nws == L.adaln_out_bwd_workspace_bytes(2, 33, 3072)
    args = [fake(i) for i in range(7)]
    assert L.adaln_f32_out_bwd(*args, fake(7), nws, 2, 33, 3072, None) == DEVICE
    assert L.adaln_f32_out_bwd(*args, fake(7), 8, 2, 33, 3072, None) == WORKSPACE
    assert L.adaln_f32_out_bwd(*args[:5], fake(0, 32), args[6], fake(7), nws, 2, 33, 3072, None) == ALIAS
    # projection backward
    nws = L.adaln_f32_proj_bwd_workspace_bytes(2, 3072)
    assert nws == 24 * 2 * 3072 * 4
    p = [fake(i) for i in range(7)]
    assert L.adaln_f32_proj_bwd(*p, 2, fake(7), nws, 2, 3072, None) == ARG
    assert L.adaln_f32_proj_bwd(*p, 0, fake(7), nws, 2, 3072, None) == DEVICE
    assert L.adaln_f32_proj_bwd(*p[:5], None, None, 0, fake(7), nws, 2, 3072, None) == DEVICE  # d_temb only
    assert L.adaln_f32_proj_bwd(*p[:5], fake(3, 64), p[6], 0, fake(7), nws, 2, 3072, None) == ALIAS


@pytest.mark.skipif(torch.cuda.is_available(), reason="a valid call with fake pointers would launch on a GPU")
def test_valid_calls_stop_at_the_device_check_without_a_gpu(L, no_gpu):
    assert proj_fwd(L) == DEVICE
    assert out_fwd(L) == DEVICE
    assert out_bwd(L) == DEVICE
    assert tree(L) == DEVICE
    assert proj_bwd(L) == DEVICE
    assert proj_bwd(L, dW_acc=None, db_acc=None, dW=None, db=None) == DEVICE


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        binding.load(str(tmp_path / "libadaln.so"))
