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

import numpy as np

REL_F32 = 1e-5


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
    return {"n": int(got.size), "exact": int((dist == 0).sum()), "ulp1": int((dist == 1).sum()),
            "floor_only": floor_only, "max_ulp": int(dist.max()) if dist.size else 0}


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
    return {"n": int(got.size), "exact": int((diff == 0).sum()), "floor_only": floor_only,
            "max_rel": float(np.max(relerr[np.isfinite(relerr)])) if np.isfinite(relerr).any() else 0.0}


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


def floor_d_emb(x_f64, g_f64):
    """d_scale = sum_s g xhat with xhat off by 2^-18 (a_row + |xhat|);
    d_shift = sum_s g: floor = 2^-16 * sum_s |g| (1 + |xhat| + a_row)."""
    a, xh, _ = row_scale(x_f64)
    g = np.abs(g_f64)
    fs = F_OUT * (g * (1.0 + np.abs(xh) + a)).sum(axis=1)
    fh = F_OUT * g.sum(axis=1)
    return np.concatenate([fs, fh], axis=1)


def floor_d_temb(e_f64, W_f64, dsilu_f64):
    """d_temb = (sum_n e W) * silu'(t): floor = 2^-16 * (sum_n |e W|) * |silu'(t)|."""
    return F_OUT * (np.abs(e_f64) @ np.abs(W_f64)) * np.abs(dsilu_f64)
