"""Comparison rules used by the parity tests.

bf16 outputs pass when they are within one bf16 ulp of the oracle's value
(distance counted in representable bf16 steps, so +0 and -0 are equal), or,
where the computed quantity cancels, when the absolute difference is within
an error-bound floor derived from the fp32 arithmetic that produces it.

fp32 outputs pass when the relative difference is at most 1e-5, or when the
absolute difference is within the floor.

Every rule returns the number of elements that passed only through the floor,
so the tests can report it.
"""

from __future__ import annotations

import json
import os

import numpy as np

REL_F32 = 1e-5


def _report(kind, what, stats):
    """Print the comparison statistics and, when ADALN_PARITY_LOG names a file,
    append them to it as one JSON line (the floor-only counts are reported
    per check)."""
    line = {"check": kind, "what": what, **stats}
    print("PARITY " + json.dumps(line))
    path = os.environ.get("ADALN_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(line) + "\n")


def bf16_to_f64(h):
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def bf16_ord(h):
    """Signed position of a bf16 value on the number line (+0 and -0 -> 0)."""
    h = np.asarray(h, dtype=np.uint16).astype(np.int64)
    mag = h & 0x7FFF
    return np.where(h & 0x8000, -mag, mag)


def bf16_ulp_dist(a, b):
    return np.abs(bf16_ord(a) - bf16_ord(b))


def check_bf16(got, want, floor=None, max_ulp=1, what="bf16"):
    """Assert got (bf16 bits) is within ``max_ulp`` of want or within ``floor``.

    Returns a dict of statistics: exact matches, 1-ulp, floor-only passes."""
    got = np.asarray(got, dtype=np.uint16)
    want = np.asarray(want, dtype=np.uint16)
    assert got.shape == want.shape, (got.shape, want.shape)
    dist = bf16_ulp_dist(got, want)
    ok = dist <= max_ulp
    floor_only = 0
    if floor is not None:
        diff = np.abs(bf16_to_f64(got) - bf16_to_f64(want))
        by_floor = (~ok) & (diff <= np.broadcast_to(floor, diff.shape))
        floor_only = int(by_floor.sum())
        ok = ok | by_floor
    bad = np.flatnonzero(~ok)
    if len(bad):
        i = bad[0]
        msg = (f"{what}: {len(bad)} of {got.size} elements out of tolerance; first at flat index {i}: "
               f"got {bf16_to_f64(got.reshape(-1)[i:i+1])[0]!r} want {bf16_to_f64(want.reshape(-1)[i:i+1])[0]!r} "
               f"({int(dist.reshape(-1)[i])} ulp)")
        if floor is not None:
            msg += f" floor {np.broadcast_to(floor, got.shape).reshape(-1)[i]!r}"
        raise AssertionError(msg)
    stats = {"n": int(got.size), "exact": int((dist == 0).sum()), "ulp1": int((dist == 1).sum()),
             "floor_only": floor_only, "max_ulp": int(dist.max()) if dist.size else 0}
    _report("bf16", what, stats)
    return stats


def check_f32(got, want, floor=None, rel=REL_F32, what="fp32"):
    """Assert |got - want| <= rel*|want| or <= floor, elementwise."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    diff = np.abs(got - want)
    ok = diff <= rel * np.abs(want)
    floor_only = 0
    if floor is not None:
        by_floor = (~ok) & (diff <= np.broadcast_to(floor, diff.shape))
        floor_only = int(by_floor.sum())
        ok = ok | by_floor
    bad = np.flatnonzero(~ok)
    if len(bad):
        i = bad[0]
        raise AssertionError(
            f"{what}: {len(bad)} of {got.size} elements out of tolerance; first at flat index {i}: "
            f"got {got.reshape(-1)[i]!r} want {want.reshape(-1)[i]!r} rel {diff.reshape(-1)[i] / max(abs(want.reshape(-1)[i]), 1e-300):.3g}"
            + (f" floor {np.broadcast_to(floor, got.shape).reshape(-1)[i]!r}" if floor is not None else ""))
    with np.errstate(divide="ignore", invalid="ignore"):
        relerr = np.where(want != 0, diff / np.abs(want), np.where(diff == 0, 0.0, np.inf))
    stats = {"n": int(got.size), "exact": int((diff == 0).sum()), "floor_only": floor_only,
             "max_rel": float(np.max(relerr[np.isfinite(relerr)])) if np.isfinite(relerr).any() else 0.0}
    _report("f32", what, stats)
    return stats


def assert_bitwise(got, want, what="bitwise"):
    """Assert two arrays hold the same bytes (same shape and dtype)."""
    got = np.ascontiguousarray(got)
    want = np.ascontiguousarray(want)
    assert got.shape == want.shape and got.dtype == want.dtype, (what, got.shape, got.dtype, want.shape, want.dtype)
    u = {1: np.uint8, 2: np.uint16, 4: np.uint32, 8: np.uint64}[got.itemsize]
    gv = got.reshape(-1).view(u)
    wv = want.reshape(-1).view(u)
    bad = np.flatnonzero(gv != wv)
    if len(bad):
        i = int(bad[0])
        raise AssertionError(f"{what}: {len(bad)} of {got.size} elements differ bitwise; first at flat index {i}: "
                             f"got {got.reshape(-1)[i]!r} want {want.reshape(-1)[i]!r}")


# ---------------------------------------------------------------------------
# error-bound floors
#
# The CUDA kernels compute row statistics with fp32 sums of at most a few
# dozen sequential terms per thread followed by fixed shuffle/shared-memory
# trees; with D <= 8192 the depth of any fp32 reduction is below 64, so the
# relative error of a sum is below 64 * 2^-24 = 2^-18 of the sum of the
# absolute values of its terms.  The floors below take that bound (2^-18) for
# every reduction, and 2^-16 (four times it) for quantities built from two or
# three of them; the factor of four also covers the fp32 roundings of the
# elementwise steps that follow.
# ---------------------------------------------------------------------------

F_RED = 2.0 ** -18
F_OUT = 2.0 ** -16


def row_scale(x_f64):
    """a_row = mean_d |x| * rstd: the size of the error of (x - mean) * rstd
    coming from the error of the mean, per unit of 2^-18."""
    x = np.asarray(x_f64, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + 1e-6)
    return np.abs(x).mean(axis=-1, keepdims=True) * rstd, (x - mu) * rstd, rstd


def floor_emb(u_f64, W_f64, b_f64):
    """emb[b,n] = sum_k u W + bias in fp32: floor = 2^-16 * (sum_k |u W| + |bias|)."""
    return F_OUT * (np.abs(u_f64) @ np.abs(W_f64).T + np.abs(b_f64)[None, :])


def floor_out(x_f64, onep_f64, shift_f64):
    """out = xhat*onep + shift, xhat carrying an absolute error below
    2^-18 * (a_row + |xhat|): floor = 2^-16 * ((a_row + |xhat|) |onep| + |xhat onep| + |shift|)."""
    a, xh, _ = row_scale(x_f64)
    on = onep_f64[:, None, :]
    sh = shift_f64[:, None, :]
    return F_OUT * ((a + np.abs(xh)) * np.abs(on) + np.abs(xh * on) + np.abs(sh))


def floor_dx(x_f64, g_f64, onep_f64):
    """dx = rstd (gh - mean(gh) - xhat mean(gh xhat)), gh = g*onep:
    floor = 2^-16 * rstd * (|gh| + mean|gh| + (|xhat| + a_row) * mean(|gh| (|xhat| + a_row)))."""
    a, xh, rstd = row_scale(x_f64)
    gh = np.abs(g_f64 * onep_f64[:, None, :])
    w = np.abs(xh) + a
    return F_OUT * rstd * (gh + gh.mean(axis=-1, keepdims=True) + w * (gh * w).mean(axis=-1, keepdims=True))


# The fixed 32-way tree with Neumaier tiles stays within 2^-23 |sum| +
# 2^-30 sum|x| of the exact sum (the compensated-summation bound 2u|s| +
# O(n u^2) sum|x| with n <= 2^18 tokens; checked on the oracle's fp32 replay of
# the tree, to which the GPU result is bitwise equal, where a plain tree breaks
# it); the oracle's value is the exact sum rounded once to fp32 (2^-24 |sum|).
# The floor takes twice their total.
F_TREE_REL = 2.0 ** -22
F_TREE_ABS = 2.0 ** -29


def floor_d_emb(x_f64, g_f64):
    """d_scale = sum_s g xhat with xhat off by 2^-18 (a_row + |xhat|):
    floor = 2^-16 * sum_s |g| (1 + |xhat| + a_row).  d_shift = sum_s g carries
    no xhat error, only the tree's: floor = 2^-22 |sum_s g| + 2^-29 sum_s |g|."""
    a, xh, _ = row_scale(x_f64)
    g = np.abs(g_f64)
    fs = F_OUT * (g * (1.0 + np.abs(xh) + a)).sum(axis=1)
    fh = F_TREE_REL * np.abs(np.asarray(g_f64).sum(axis=1)) + F_TREE_ABS * g.sum(axis=1)
    return np.concatenate([fs, fh], axis=1)


def floor_d_temb(e_f64, W_f64, dsilu_f64):
    """d_temb = (sum_n e W) * silu'(t): floor = 2^-16 * (sum_n |e W|) * |silu'(t)|."""
    return F_OUT * (np.abs(e_f64) @ np.abs(W_f64)) * np.abs(dsilu_f64)


def check_rows(inp_x, inp_dy, emb, got, orc, what, max_floor_frac=1e-5, rows_per_chunk=512):
    """out, mean, rstd and dx of every token row against the oracle (fed the
    GPU's emb, the staged reading), in chunks of rows so that the fp64 floors
    stay small in memory.  Asserts that at most max_floor_frac of the elements
    pass only through their error-bound floor.  Returns the summed statistics."""
    B, S, D = inp_x.shape
    tot = {k: {"n": 0, "exact": 0, "ulp1": 0, "floor_only": 0, "max_ulp": 0} for k in ("out", "dx")}
    for b in range(B):
        e = emb[b:b + 1]
        onep = bf16_to_f64(_bf16_of(np.float32(1) + bf16_to_f64(e[:, :D]).astype(np.float32)))
        shift = bf16_to_f64(e[:, D:])
        for s0 in range(0, S, rows_per_chunk):
            s1 = min(S, s0 + rows_per_chunk)
            x = np.ascontiguousarray(inp_x[b:b + 1, s0:s1])
            dy = np.ascontiguousarray(inp_dy[b:b + 1, s0:s1])
            w_out, w_mean, w_rstd = orc.out_fwd(x, e)
            w_dx, _ = orc.out_bwd(dy, x, e)
            xf = bf16_to_f64(x)
            st_o = _quiet(check_bf16, got["out"][b:b + 1, s0:s1], w_out, floor_out(xf, onep, shift),
                          what=f"{what}: out")
            _quiet(check_f32, got["mean"][b:b + 1, s0:s1], w_mean, F_RED * np.abs(xf).mean(-1), what=f"{what}: mean")
            _quiet(check_f32, got["rstd"][b:b + 1, s0:s1], w_rstd, what=f"{what}: rstd")
            st_d = _quiet(check_bf16, got["dx"][b:b + 1, s0:s1], w_dx, floor_dx(xf, bf16_to_f64(dy), onep),
                          what=f"{what}: dx")
            for k, st in (("out", st_o), ("dx", st_d)):
                for f in ("n", "exact", "ulp1", "floor_only"):
                    tot[k][f] += st[f]
                tot[k]["max_ulp"] = max(tot[k]["max_ulp"], st["max_ulp"])
    for k in ("out", "dx"):
        _report("bf16", f"{what}: {k} (all {B * S} rows)", tot[k])
        assert tot[k]["floor_only"] <= max_floor_frac * tot[k]["n"], (k, tot[k])
    return tot


def _bf16_of(a):
    """fp32 values -> bf16 bits, round to nearest even (numpy, exact)."""
    u = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def _quiet(fn, *args, **kw):
    """Run a check without its per-call report (the caller reports totals)."""
    global _report
    saved = _report
    _report = lambda *a, **k: None
    try:
        return fn(*args, **kw)
    finally:
        _report = saved
