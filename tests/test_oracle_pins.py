"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test ties one oracle function to one of: a value the pages print (the
token-tree cancellation result, the SiLU derivative at 1), exact rational
arithmetic on small inputs, an independent library routine (PyTorch's fp64
LayerNorm, linear, SiLU and autograd on the CPU; math.fsum), a closed form or
an invariant of the mathematics, or finite differences.  They are chosen so
that a dropped term, a wrong sign or index, a transposed operand, a missing
rounding point or a swapped (scale, shift) order fails at least one of them.
"""

from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from invariant_dit_adaln_gb300 import synth
from tolerance import assert_bitwise, bf16_to_f64, bf16_ulp_dist

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
EPS32 = float(np.float32(1e-6))


def golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------------------
# exact bf16 rounding, written with rationals (independent of the oracle's)
# ---------------------------------------------------------------------------

def bf16_exact_round(v: Fraction) -> int:
    """Bits of the bf16 nearest to the rational v (ties to even)."""
    if v == 0:
        return 0
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    # a in [2^e, 2^(e+1)); spacing 2^(e-7) for normals, 2^-133 below 2^-126
    q = max(e - 7, -133)
    scaled = a / (Fraction(2) ** q)
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    val = Fraction(n) * Fraction(2) ** q
    f = np.float32(float(val))
    assert Fraction(float(f)) == val
    return sign | int(np.array([f], dtype=np.float32).view(np.uint32)[0] >> 16)


def test_bf16_rounding_from_f64_matches_exact(orc):
    rng = np.random.default_rng(1)
    vals = list(rng.standard_normal(3000) * np.exp2(rng.integers(-140, 120, 3000)))
    # ties and near-ties, subnormals, zeros
    for k in range(0, 256, 7):
        base = 1.0 + k / 128.0
        vals += [base + 1 / 256.0, -(base + 1 / 256.0), np.nextafter(base + 1 / 256.0, 10), np.nextafter(base + 1 / 256.0, 0)]
    vals += [2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -135, 2.0 ** -126 * 1.5, 0.0, -0.0, 2.0 ** 127 * 1.9921875]
    x = np.array(vals, dtype=np.float64)
    got = orc.bf16_from_f64(x)
    want = np.array([bf16_exact_round(Fraction(float(v))) if v != 0 else (0x8000 if math.copysign(1, v) < 0 else 0)
                     for v in x], dtype=np.uint16)
    assert_bitwise(got, want, "bf16 from fp64")


# ---------------------------------------------------------------------------
# SiLU and its derivative
# ---------------------------------------------------------------------------

def test_silu_derivative_worked_value(orc):
    (t, want, tol), = golden_rows("silu_vjp.txt")
    got = orc.dsilu_f64(np.array([float(t)]))[0]
    assert abs(got - float(want)) <= float(tol)
    # and the derivative is the derivative: central differences of t*sigmoid(t)
    ts = np.linspace(-8, 8, 33)
    h = 1e-6
    fd = ((ts + h) / (1 + np.exp(-(ts + h))) - (ts - h) / (1 + np.exp(-(ts - h)))) / (2 * h)
    np.testing.assert_allclose(orc.dsilu_f64(ts), fd, rtol=1e-8, atol=1e-9)


def test_silu_bf16_is_nearest_bf16_of_exact_silu(orc):
    import mpmath
    mpmath.mp.prec = 200
    # every bf16 with |t| in a useful range, sampled; plus the extremes
    all_bits = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    fin = all_bits[(all_bits & 0x7F80) != 0x7F80]
    rng = np.random.default_rng(2)
    pick = np.concatenate([rng.choice(fin, 3000, replace=False),
                           np.array([0x0000, 0x8000, 0x3F80, 0xBF80, 0x0001, 0x8001, 0x7F7F, 0xFF7F], np.uint16)])
    got = orc.silu_bf16(pick)
    want = []
    for h in pick:
        t = mpmath.mpf(float(bf16_to_f64(np.array([h]))[0]))
        s = t / (1 + mpmath.exp(-t))
        if abs(s) < mpmath.mpf(2) ** -135:  # below half the smallest bf16 subnormal
            want.append(0x8000 if t < 0 else 0)
        else:
            mag = Fraction(int(s.man)) * Fraction(2) ** int(s.exp)  # mpmath keeps the sign apart
            want.append(bf16_exact_round(-mag if s < 0 else mag))
    want = np.array(want, dtype=np.uint16)
    # The oracle rounds the fp64 value of t / (1 + exp(-t)).  For |t| < 2^-125
    # that value is t/2 exactly (the t^2/4 term is below fp64 resolution) and
    # falls in the bf16 subnormal range, where an odd t makes it a bf16 tie; the
    # exact value lies just off the tie.  Those inputs are the only ones allowed
    # to differ, by one ulp.
    subnormal = (pick & 0x7F80) <= 0x0080
    dist = bf16_ulp_dist(got, want)  # +0 and -0 count as equal
    mism = np.flatnonzero(dist != 0)
    assert np.all(subnormal[mism]), [(hex(pick[i]), hex(got[i]), hex(want[i])) for i in mism[:5]]
    assert np.all(dist[mism] == 1)
    t = bf16_to_f64(pick[subnormal])
    assert_bitwise(got[subnormal], orc.bf16_from_f64(t / 2.0), "tiny t: u = bf16(t/2)")


# ---------------------------------------------------------------------------
# projection forward
# ---------------------------------------------------------------------------

def _bf16(a):
    return synth.bf16_bits_from_f32(np.asarray(a, dtype=np.float32))


def test_proj_fwd_exact_rational_small(orc):
    """emb must be the nearest bf16 of the exact sum u.W + b, u = bf16(silu(t))."""
    rng = np.random.default_rng(3)
    B, D = 2, 16
    temb = _bf16(rng.standard_normal((B, D)))
    W = _bf16(rng.standard_normal((2 * D, D)) * 0.3)
    b = _bf16(rng.standard_normal(2 * D) * 0.3)
    u = orc.silu_bf16(temb)  # pinned above
    uf = bf16_to_f64(u)
    Wf = bf16_to_f64(W)
    bf = bf16_to_f64(b)
    got = orc.proj_fwd(temb, W, b)
    for i in range(B):
        for n in range(2 * D):
            exact = sum(Fraction(float(uf[i, k])) * Fraction(float(Wf[n, k])) for k in range(D)) + Fraction(float(bf[n]))
            assert got[i, n] == bf16_exact_round(exact) if exact != 0 else True, (i, n)


def test_proj_fwd_special_cases_and_order(orc):
    rng = np.random.default_rng(4)
    B, D = 3, 32
    temb = _bf16(rng.standard_normal((B, D)))
    W = _bf16(rng.standard_normal((2 * D, D)) * 0.02)
    b = _bf16(rng.standard_normal(2 * D) * 0.02)
    # W = 0 -> emb = b bitwise
    assert_bitwise(orc.proj_fwd(temb, np.zeros_like(W), b), np.broadcast_to(b, (B, 2 * D)), "W=0")
    # temb = 0 -> silu = 0 -> emb = b
    assert_bitwise(orc.proj_fwd(np.zeros_like(temb), W, b), np.broadcast_to(b, (B, 2 * D)), "temb=0")
    # (scale, shift) order: zeroing the second half of W leaves emb[:, D:] = b[D:]
    W2 = W.copy()
    W2[D:] = 0
    e2 = orc.proj_fwd(temb, W2, b)
    assert_bitwise(e2[:, D:], np.broadcast_to(b[D:], (B, D)), "shift half")
    assert_bitwise(e2[:, :D], orc.proj_fwd(temb, W, b)[:, :D], "scale half")


def test_proj_fwd_f64_matches_torch(orc):
    rng = np.random.default_rng(5)
    B, D = 3, 24
    temb = rng.standard_normal((B, D))
    W = rng.standard_normal((2 * D, D)) * 0.1
    b = rng.standard_normal(2 * D) * 0.1
    ref = torch.nn.functional.linear(torch.nn.functional.silu(torch.from_numpy(temb)),
                                     torch.from_numpy(W), torch.from_numpy(b)).numpy()
    np.testing.assert_allclose(orc.proj_fwd_f64(temb, W, b), ref, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------------------
# LayerNorm + modulation forward
# ---------------------------------------------------------------------------

def test_out_fwd_f64_matches_torch(orc):
    rng = np.random.default_rng(6)
    B, S, D = 2, 5, 40
    x = rng.standard_normal((B, S, D)) * 3 + 0.5
    x[1, 2] *= 50
    scale = rng.standard_normal((B, D)) * 0.1
    shift = rng.standard_normal((B, D)) * 0.1
    tx = torch.from_numpy(x)
    ref = (torch.nn.functional.layer_norm(tx, (D,), eps=1e-6) * (1 + torch.from_numpy(scale)[:, None, :])
           + torch.from_numpy(shift)[:, None, :]).numpy()
    np.testing.assert_allclose(orc.out_fwd_f64(x, scale, shift, 1e-6), ref, rtol=1e-11, atol=1e-12)


def test_out_fwd_reduces_to_plain_layernorm_when_W_and_b_are_zero(orc):
    """W = b = 0 -> emb = 0 -> onep = 1, shift = 0 -> out = bf16(fp32(LN(x)))."""
    rng = np.random.default_rng(7)
    B, S, D = 2, 7, 64
    x = _bf16(rng.standard_normal((B, S, D)) * 2)
    emb = orc.proj_fwd(_bf16(rng.standard_normal((B, D))), np.zeros((2 * D, D), np.uint16), np.zeros(2 * D, np.uint16))
    assert not emb.any()
    out, mean, rstd = orc.out_fwd(x, emb)
    xf = torch.from_numpy(bf16_to_f64(x))
    ln = torch.nn.functional.layer_norm(xf, (D,), eps=EPS32).numpy()
    want = synth.bf16_bits_from_f32(ln.astype(np.float32))
    assert_bitwise(out, want, "plain LN")
    np.testing.assert_array_equal(mean, xf.mean(-1).numpy().astype(np.float32))
    var = xf.var(-1, unbiased=False).numpy()
    np.testing.assert_array_equal(rstd, (1.0 / np.sqrt(var + EPS32)).astype(np.float32))


def test_out_fwd_invariants(orc):
    rng = np.random.default_rng(8)
    B, S, D = 1, 4, 256
    x = rng.standard_normal((B, S, D)) * 4 - 1
    xh = orc.out_fwd_f64(x, np.zeros((B, D)), np.zeros((B, D)), 1e-6)
    var = x.var(-1)
    np.testing.assert_allclose(xh.mean(-1), 0, atol=1e-13)
    np.testing.assert_allclose(xh.var(-1), var / (var + 1e-6), rtol=1e-12)
    # constant row -> xhat = 0 exactly -> out = shift bitwise
    xc = np.full((1, 3, D), 0x3FC0, np.uint16)  # 1.5
    emb = _bf16(rng.standard_normal((1, 2 * D)))
    out, mean, rstd = orc.out_fwd(xc, emb)
    assert_bitwise(out, np.broadcast_to(emb[:, D:], (1, 3, D)).astype(np.uint16), "constant row")
    assert np.all(mean == 1.5)


def _pm_one_row(D):
    return np.tile(np.array([0xBF80, 0x3F80], np.uint16), D // 2)  # -1, +1, ...: mean 0, var 1


def test_out_fwd_rounding_point_onep(orc):
    """Worked example of '(1 + scale) rounds once in bf16'.

    x = (-1, +1, ...): mean 0, variance 1, xhat = +-1/sqrt(1 + eps) = +-0.99999952
    (fp32).  bf16 values in [1, 2) are 2^-7 apart.  scale = 3 * 2^-8: 1 + scale =
    1.01171875 is the midpoint of 1 + 2^-7 and 1 + 2^-6; ties-to-even gives
    onep = 1 + 2^-6.  With shift = 0, m = 0.99999952 * 1.015625 = 1.0156245,
    so out = 1 + 2^-6 on the +1 entries.  Without the rounding of (1 + scale),
    m = 0.99999952 * 1.01171875 = 1.0117183 lies below the midpoint and out
    would be 1 + 2^-7."""
    D = 8
    x = _pm_one_row(D).reshape(1, 1, D)
    emb = np.zeros((1, 2 * D), np.uint16)
    emb[0, :D] = _bf16(np.full(D, 3 * 2.0 ** -8))
    assert np.all(bf16_to_f64(emb[0, :D]) == 3 * 2.0 ** -8)
    out, _, _ = orc.out_fwd(x, emb)
    vals = bf16_to_f64(out[0, 0])
    assert np.all(vals[1::2] == 1 + 2.0 ** -6), vals
    assert np.all(vals[0::2] == -(1 + 2.0 ** -6)), vals


def test_out_fwd_rounding_point_fp32_modulation(orc):
    """Worked example of 'the modulation promotes to fp32, one bf16 store'.

    xhat = 0.99999952, onep = 1 (scale 0), shift = 3 * 2^-8: m = 1.0117183 (fp32)
    lies below the bf16 midpoint 1.01171875, so out = 1 + 2^-7.  Rounding
    xhat * onep to bf16 first (1.0) would make m = 1.01171875, a tie, and out
    would be 1 + 2^-6."""
    D = 8
    x = _pm_one_row(D).reshape(1, 1, D)
    emb = np.zeros((1, 2 * D), np.uint16)
    emb[0, D:] = _bf16(np.full(D, 3 * 2.0 ** -8))
    out, _, _ = orc.out_fwd(x, emb)
    vals = bf16_to_f64(out[0, 0])
    assert np.all(vals[1::2] == 1 + 2.0 ** -7), vals


# ---------------------------------------------------------------------------
# LayerNorm + modulation backward
# ---------------------------------------------------------------------------

def _torch_out_bwd(dy, x, scale, eps):
    tx = torch.from_numpy(x).requires_grad_(True)
    ts = torch.from_numpy(scale).requires_grad_(True)
    th = torch.zeros_like(ts).requires_grad_(True)
    D = x.shape[-1]
    out = torch.nn.functional.layer_norm(tx, (D,), eps=eps) * (1 + ts[:, None, :]) + th[:, None, :]
    out.backward(torch.from_numpy(dy))
    return tx.grad.numpy(), ts.grad.numpy(), th.grad.numpy()


def test_out_bwd_f64_matches_torch_autograd(orc):
    rng = np.random.default_rng(9)
    B, S, D = 2, 6, 48
    x = rng.standard_normal((B, S, D)) * 2
    x[0, 3] *= 50
    scale = rng.standard_normal((B, D)) * 0.2
    dy = rng.standard_normal((B, S, D))
    dx, ds, dh = orc.out_bwd_f64(dy, x, scale, 1e-6)
    rdx, rds, rdh = _torch_out_bwd(dy, x, scale, 1e-6)
    np.testing.assert_allclose(dx, rdx, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(ds, rds, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dh, rdh, rtol=1e-12, atol=1e-12)


def test_out_bwd_f64_finite_differences(orc):
    rng = np.random.default_rng(10)
    B, S, D = 1, 3, 8
    x = rng.standard_normal((B, S, D))
    scale = rng.standard_normal((B, D)) * 0.3
    shift = rng.standard_normal((B, D)) * 0.3
    dy = rng.standard_normal((B, S, D))
    dx, ds, dh = orc.out_bwd_f64(dy, x, scale, 1e-6)
    f = lambda xx, sc, sh: float((orc.out_fwd_f64(xx, sc, sh, 1e-6) * dy).sum())
    h = 1e-6
    for idx in [(0, 0, 0), (0, 1, 5), (0, 2, 7)]:
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        assert abs((f(xp, scale, shift) - f(xm, scale, shift)) / (2 * h) - dx[idx]) < 1e-6
    for j in [0, 3, 7]:
        sp, sm = scale.copy(), scale.copy()
        sp[0, j] += h
        sm[0, j] -= h
        assert abs((f(x, sp, shift) - f(x, sm, shift)) / (2 * h) - ds[0, j]) < 1e-6
        hp, hm = shift.copy(), shift.copy()
        hp[0, j] += h
        hm[0, j] -= h
        assert abs((f(x, scale, hp) - f(x, scale, hm)) / (2 * h) - dh[0, j]) < 1e-6


def test_out_bwd_dx_invariants(orc):
    """sum_d dx = 0 and sum_d dx * xhat = rstd * D * c2 * eps / (var + eps)
    (c2 = mean(gh * xhat)), for every row."""
    rng = np.random.default_rng(11)
    B, S, D = 1, 4, 128
    x = rng.standard_normal((B, S, D)) * 0.01  # small variance: eps matters
    scale = rng.standard_normal((B, D)) * 0.1
    dy = rng.standard_normal((B, S, D))
    dx, _, _ = orc.out_bwd_f64(dy, x, scale, 1e-6)
    mu = x.mean(-1, keepdims=True)
    var = x.var(-1, keepdims=True)
    r = 1 / np.sqrt(var + 1e-6)
    xh = (x - mu) * r
    gh = dy * (1 + scale[:, None, :])
    c2 = (gh * xh).mean(-1, keepdims=True)
    np.testing.assert_allclose(dx.sum(-1), 0, atol=1e-9)
    np.testing.assert_allclose((dx * xh).sum(-1, keepdims=True), r * D * c2 * 1e-6 / (var + 1e-6), rtol=1e-6, atol=1e-9)


def test_out_bwd_token_sums_are_exact(orc):
    """d_shift = sum_s dy (correctly rounded, math.fsum) and
    d_scale = sum_s dy * fp32(LN(x)) (correctly rounded), per column."""
    rng = np.random.default_rng(12)
    B, S, D = 2, 70, 16
    x = _bf16(rng.standard_normal((B, S, D)))
    dy = _bf16(rng.standard_normal((B, S, D)))
    emb = _bf16(rng.standard_normal((B, 2 * D)) * 0.1)
    _, d_emb = orc.out_bwd(dy, x, emb)
    g = bf16_to_f64(dy)
    xh = torch.nn.functional.layer_norm(torch.from_numpy(bf16_to_f64(x)), (D,), eps=EPS32).numpy().astype(np.float32)
    for b in range(B):
        for d in range(D):
            assert d_emb[b, D + d] == np.float32(math.fsum(g[b, :, d]))
            assert d_emb[b, d] == np.float32(math.fsum(g[b, :, d] * xh[b, :, d].astype(np.float64)))


def test_out_bwd_bf16_entry_rounds_the_f64_gradient(orc):
    """dx of the bf16 entry is the bf16 rounding of the exact gradient taken at
    onep = bf16(1 + scale), i.e. with scale' = onep - 1 in the fp64 map."""
    rng = np.random.default_rng(13)
    B, S, D = 2, 9, 64
    x = _bf16(rng.standard_normal((B, S, D)))
    dy = _bf16(rng.standard_normal((B, S, D)))
    emb = _bf16(rng.standard_normal((B, 2 * D)) * 0.3)
    dx, _ = orc.out_bwd(dy, x, emb)
    onep = bf16_to_f64(synth.bf16_bits_from_f32(np.float32(1) + bf16_to_f64(emb[:, :D]).astype(np.float32)))
    rdx, _, _ = _torch_out_bwd(bf16_to_f64(dy), bf16_to_f64(x), onep - 1.0, EPS32)
    assert_bitwise(dx, orc.bf16_from_f64(rdx), "dx = bf16(exact)")


# ---------------------------------------------------------------------------
# token sums
# ---------------------------------------------------------------------------

def _plain_tree(v):
    """Uncompensated 32-way tree in fp32 (for the contrast in the worked example)."""
    v = np.asarray(v, np.float32)
    while len(v) > 1:
        n = (len(v) + 31) // 32
        w = np.concatenate([v, np.zeros(n * 32 - len(v), np.float32)]).reshape(n, 32)
        s = w[:, 0].copy()
        for j in range(1, 32):
            s = (s + w[:, j]).astype(np.float32)
        v = s
    return v[0]


def test_token_tree_cancellation_worked_example(orc):
    for S, p, m, want, want_plain in golden_rows("token_tree_cancellation.txt"):
        S, p, m = int(S), int(p), int(m)
        a = np.ones((1, S, 1), np.float32)
        a[0, p, 0] = 2.0 ** 26
        a[0, m, 0] = -(2.0 ** 26)
        assert orc.token_tree_f32(a)[0, 0] == float(want), (p, m)
        assert orc.token_sum_f64(a)[0, 0] == float(want)
        if int(want_plain) >= 0:
            assert _plain_tree(a[0, :, 0]) == float(want_plain)


def test_token_tree_counts_every_token_once(orc):
    """Integer-valued inputs whose partial sums stay below 2^24: every fp32
    operation is exact, so the tree must give the exact sum.  A dropped,
    repeated or misplaced token, tile or child changes it."""
    rng = np.random.default_rng(14)
    for S in [1, 2, 31, 32, 33, 64, 65, 1023, 1024, 1025, 4096, 6032, 6889, 33000]:
        B, H = 2, 3
        a = rng.integers(-1000, 1000, size=(B, S, H)).astype(np.float32)
        a[:, :, 1] = np.arange(S, dtype=np.float32)[None, :] * 0 + (np.arange(S) % 97)[None, :]
        got = orc.token_tree_f32(a)
        assert_bitwise(got, a.astype(np.float64).sum(axis=1).astype(np.float32), f"S={S}")


def test_token_tree_error_bound_vs_exact(orc):
    """The compensated tree stays within 2^-23 |sum| + 2^-30 sum|x| of the exact
    sum (math.fsum) on wide-range random inputs up to S = 40000; a plain fp32
    tree exceeds that bound on the same inputs."""
    rng = np.random.default_rng(15)
    worst_plain = 0.0
    for S in [33, 1000, 4096, 6889, 40000]:
        H = 4
        a = (rng.standard_normal((1, S, H)) * np.exp2(rng.integers(-12, 12, (1, S, H)))).astype(np.float32)
        got = orc.token_tree_f32(a)[0]
        for h in range(H):
            col = a[0, :, h].astype(np.float64)
            exact = math.fsum(col)
            bound = 2.0 ** -23 * abs(exact) + 2.0 ** -30 * np.abs(col).sum()
            assert abs(float(got[h]) - exact) <= bound, (S, h, float(got[h]), exact)
            worst_plain = max(worst_plain, abs(float(_plain_tree(a[0, :, h])) - exact) / bound)
    assert worst_plain > 1.0


def test_token_tree_small_cases(orc):
    rng = np.random.default_rng(16)
    a = rng.standard_normal((3, 1, 5)).astype(np.float32)
    assert_bitwise(orc.token_tree_f32(a), a[:, 0, :], "S=1 is the identity")
    a2 = rng.standard_normal((2, 2, 7)).astype(np.float32)
    assert_bitwise(orc.token_tree_f32(a2), (a2[:, 0] + a2[:, 1]).astype(np.float32), "S=2 is one IEEE add")


def test_token_sum_f64_is_correctly_rounded(orc):
    rng = np.random.default_rng(17)
    a = (rng.standard_normal((2, 500, 3)) * np.exp2(rng.integers(-20, 20, (2, 500, 3)))).astype(np.float32)
    got = orc.token_sum_f64(a)
    for b in range(2):
        for h in range(3):
            assert got[b, h] == math.fsum(a[b, :, h].astype(np.float64))


def f32_exact_round(v: Fraction) -> Fraction:
    """The fp32 value nearest to the rational v (ties to even), as a rational."""
    if v == 0:
        return Fraction(0)
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    # a in [2^e, 2^(e+1)); spacing 2^(e-23) for normals, 2^-149 below 2^-126
    q = max(e - 23, -149)
    scaled = a / (Fraction(2) ** q)
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    r = Fraction(n) * Fraction(2) ** q
    return r if v > 0 else -r


def test_f32_exact_round_agrees_with_ieee_single():
    """The helper above against numpy's own fp32 conversion of fp64 values
    (one rounding), including ties, near-ties and subnormals."""
    rng = np.random.default_rng(30)
    vals = list(rng.standard_normal(2000) * np.exp2(rng.integers(-160, 120, 2000)))
    for k in range(1, 200, 3):
        tie = 1.0 + (2 * k + 1) * 2.0 ** -24
        vals += [tie, -tie, np.nextafter(tie, 10), np.nextafter(tie, 0)]
    vals += [2.0 ** -149, 2.0 ** -150, 3 * 2.0 ** -151, 1.5 * 2.0 ** -126]
    for v in vals:
        assert float(f32_exact_round(Fraction(float(v)))) == float(np.float32(v)), v


def test_bwd_products_two_roundings_at_nonzero_mean(orc):
    """The scale-tree product p = fp32(g * fp32(fp32(x - mean) * rstd)) from the
    forward's saved statistics, pinned bit for bit against exact rationals with
    an RNE rounding after the subtraction, after the multiply by rstd and after
    the multiply by g.  The inputs (mean with a full fp32 significand, rstd far
    from 1, and x near the mean where x - mean loses bits) are chosen so that
    the plausible wrong orders give different bits: x rstd - mean rstd, x - mean
    kept exact, and a single rounding of the exact product."""
    rng = np.random.default_rng(31)
    B, S, D = 1, 64, 64
    mean = (rng.standard_normal((B, S)) * 3 + rng.uniform(-1, 1, (B, S)) * 1e-3).astype(np.float32)
    rstd = np.exp(rng.uniform(-4, 4, (B, S))).astype(np.float32)
    near = mean[..., None] + rng.standard_normal((B, S, D)) * np.exp2(rng.integers(-12, 2, (B, S, D)))
    x = synth.bf16_bits_from_f32(near.astype(np.float32))
    dy = synth.bf16_bits_from_f32((rng.standard_normal((B, S, D)) * 2).astype(np.float32))
    got = orc.bwd_products_f32(dy, x, mean, rstd)
    xf, gf = bf16_to_f64(x), bf16_to_f64(dy)
    R = f32_exact_round
    differ = {"x*rstd - mean*rstd": 0, "x - mean exact": 0, "one rounding": 0}
    for s in range(S):
        m, r = Fraction(float(mean[0, s])), Fraction(float(rstd[0, s]))
        for d in range(D):
            xv, gv = Fraction(float(xf[0, s, d])), Fraction(float(gf[0, s, d]))
            want = R(gv * R(R(xv - m) * r))
            assert Fraction(float(got[0, s, d])) == want, (s, d)
            assert Fraction(float(got[0, s, D + d])) == gv
            differ["x*rstd - mean*rstd"] += R(gv * R(R(xv * r) - R(m * r))) != want
            differ["x - mean exact"] += R(gv * R((xv - m) * r)) != want
            differ["one rounding"] += R(gv * (xv - m) * r) != want
    # every wrong order is caught by this input set
    assert all(v > 0 for v in differ.values()), differ


def test_bwd_products_reuse_forward_statistics(orc):
    """prod = (g * fp32(fp32(x - mean) * rstd), g): with mean 0 and rstd 1 the
    product is g * x exactly; the shift half is g."""
    rng = np.random.default_rng(18)
    B, S, D = 1, 3, 8
    x = _bf16(rng.standard_normal((B, S, D)))
    dy = _bf16(rng.standard_normal((B, S, D)))
    p = orc.bwd_products_f32(dy, x, np.zeros((B, S), np.float32), np.ones((B, S), np.float32))
    assert_bitwise(p[..., :D], (bf16_to_f64(dy) * bf16_to_f64(x)).astype(np.float32), "scale products")
    assert_bitwise(p[..., D:], bf16_to_f64(dy).astype(np.float32), "shift products")


# ---------------------------------------------------------------------------
# projection backward
# ---------------------------------------------------------------------------

def test_proj_bwd_f64_matches_torch_autograd(orc):
    rng = np.random.default_rng(19)
    B, D = 3, 16
    temb = rng.standard_normal((B, D))
    W = rng.standard_normal((2 * D, D)) * 0.2
    b = rng.standard_normal(2 * D) * 0.2
    de = rng.standard_normal((B, 2 * D))
    tt = torch.from_numpy(temb).requires_grad_(True)
    tW = torch.from_numpy(W).requires_grad_(True)
    tb = torch.from_numpy(b).requires_grad_(True)
    torch.nn.functional.linear(torch.nn.functional.silu(tt), tW, tb).backward(torch.from_numpy(de))
    d_temb, dW, db = orc.proj_bwd_f64(de, temb, W)
    np.testing.assert_allclose(d_temb, tt.grad.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dW, tW.grad.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(db, tb.grad.numpy(), rtol=1e-12, atol=1e-13)


def test_proj_bwd_bf16_entry(orc):
    """d_temb = bf16(exact (e @ W) * silu'(t)) with e = bf16(d_emb) (torch fp64
    autograd of linear(silu)); dW = sum_b e u with u = bf16(silu(t)); B = 1
    gives dW = e (x) u exactly."""
    rng = np.random.default_rng(20)
    B, D = 2, 32
    temb = _bf16(rng.standard_normal((B, D)))
    W = _bf16(rng.standard_normal((2 * D, D)) * 0.05)
    d_emb = rng.standard_normal((B, 2 * D)).astype(np.float32) * 3
    d_temb, dW, db = orc.proj_bwd(d_emb, temb, W)
    e = bf16_to_f64(synth.bf16_bits_from_f32(d_emb))
    tt = torch.from_numpy(bf16_to_f64(temb)).requires_grad_(True)
    torch.nn.functional.linear(torch.nn.functional.silu(tt), torch.from_numpy(bf16_to_f64(W))).backward(torch.from_numpy(e))
    assert_bitwise(d_temb, orc.bf16_from_f64(tt.grad.numpy()), "d_temb")
    u = bf16_to_f64(orc.silu_bf16(temb))
    np.testing.assert_allclose(dW, e.T @ u, rtol=1e-15, atol=0)
    np.testing.assert_array_equal(db, e.sum(0))
    d1, dW1, db1 = orc.proj_bwd(d_emb[:1], temb[:1], W)
    np.testing.assert_array_equal(dW1, np.outer(e[0], u[0]))


def test_wgrad_seq_f32_order_and_chunking(orc):
    """Sequential fp32 accumulation over samples: B = 1 is the exact outer
    product; the 5 chunkings of a workload give identical bytes; appended
    zero samples change nothing; the result is within the sequential-sum
    bound (B - 1) * 2^-24 * sum|terms| of the fp64 value."""
    rng = np.random.default_rng(21)
    B, D = 12, 16
    temb = _bf16(rng.standard_normal((B, D)))
    d_emb = rng.standard_normal((B, 2 * D)).astype(np.float32)
    W = _bf16(rng.standard_normal((2 * D, D)) * 0.05)
    e = bf16_to_f64(synth.bf16_bits_from_f32(d_emb))
    u = bf16_to_f64(orc.silu_bf16(temb))
    dW1, db1 = orc.wgrad_seq_f32(d_emb[:1], temb[:1])
    assert_bitwise(dW1, np.outer(e[0], u[0]).astype(np.float32), "B=1")
    full, fullb = orc.wgrad_seq_f32(d_emb, temb)
    for chunk in [1, 2, 3, 4, 6, 12]:
        acc, accb = None, None
        for i in range(0, B, chunk):
            acc, accb = orc.wgrad_seq_f32(d_emb[i:i + chunk], temb[i:i + chunk], acc, accb, accumulate=acc is not None)
        assert_bitwise(acc, full, f"chunk {chunk}")
        assert_bitwise(accb, fullb, f"chunk {chunk} db")
    pad, padb = orc.wgrad_seq_f32(np.zeros((3, 2 * D), np.float32), temb[:3], full, fullb, accumulate=True)
    assert_bitwise(pad, full, "zero padding")
    assert_bitwise(padb, fullb, "zero padding db")
    _, dW64, db64 = orc.proj_bwd(d_emb, temb, W)
    bound = (B - 1) * 2.0 ** -24 * (np.abs(e).T @ np.abs(u))
    assert np.all(np.abs(full - dW64) <= bound + 1e-30)


def test_wgrad_seq_f32_rows(orc):
    """The sampled-rows form: B = 1 gives the exact outer product of the
    listed rows; with many samples, the listed rows of the full sequential
    accumulation, bit for bit."""
    rng = np.random.default_rng(22)
    B, D = 9, 24
    temb = _bf16(rng.standard_normal((B, D)))
    d_emb = rng.standard_normal((B, 2 * D)).astype(np.float32)
    rows = np.array([0, 5, 2 * D - 1, 17, 5], np.int32)
    e = bf16_to_f64(synth.bf16_bits_from_f32(d_emb))
    u = bf16_to_f64(orc.silu_bf16(temb))
    dW1, db1 = orc.wgrad_seq_f32_rows(d_emb[:1], temb[:1], rows)
    assert_bitwise(dW1, np.outer(e[0, rows], u[0]).astype(np.float32), "B=1 rows")
    assert_bitwise(db1, e[0, rows].astype(np.float32), "B=1 db rows")
    full, fullb = orc.wgrad_seq_f32(d_emb, temb)
    got, gotb = orc.wgrad_seq_f32_rows(d_emb, temb, rows)
    assert_bitwise(got, full[rows], "rows of the full accumulation")
    assert_bitwise(gotb, fullb[rows], "rows of db")


# ---------------------------------------------------------------------------
# block-level modulated norm with a gated residual (ScaleResidualLayerNorm-
# ScaleShift; miles_diffusion PR 108 Summary, root cause 1)
# ---------------------------------------------------------------------------

def _block(B, S, D, seed):
    return synth.make_block_inputs(B, S, D, seed)


def _tbf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def _bits_of(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_res_fwd_residual_is_eager_bf16(orc):
    """r = residual + gate * x in eager bf16: against PyTorch's bf16 ops on the
    CPU and against exact rationals rounded twice (after the product and after
    the sum); out, mean, rstd are the norm_out forward of r."""
    B, S, D = 2, 7, 40
    i = _block(B, S, D, 3)
    r, out, mean, rstd = orc.res_fwd(i["x"], i["residual"], i["gate"], i["emb"])
    t = _tbf16(i["residual"]) + _tbf16(i["gate"])[:, None, :] * _tbf16(i["x"])
    assert_bitwise(r, _bits_of(t), "r vs torch bf16")
    xf, rf, gf = bf16_to_f64(i["x"]), bf16_to_f64(i["residual"]), bf16_to_f64(i["gate"])
    one_rounding_differs = 0
    for b in range(B):
        for s in range(S):
            for d in range(D):
                p = Fraction(float(gf[b, d])) * Fraction(float(xf[b, s, d]))
                h = bf16_exact_round(p)
                hv = Fraction(float(bf16_to_f64(np.array([h], np.uint16))[0]))
                want = bf16_exact_round(Fraction(float(rf[b, s, d])) + hv)
                assert int(r[b, s, d]) == want, (b, s, d)
                one_rounding_differs += bf16_exact_round(Fraction(float(rf[b, s, d])) + p) != want
    # the product's own rounding matters on these inputs: a fused form would fail
    assert one_rounding_differs > 0
    w_out, w_mean, w_rstd = orc.out_fwd(r, i["emb"])
    assert_bitwise(out, w_out, "out")
    assert_bitwise(mean, w_mean, "mean")
    assert_bitwise(rstd, w_rstd, "rstd")


def test_res_fwd_special_cases(orc):
    """gate = 0 gives r = residual; residual = 0 gives r = bf16(gate * x);
    gate = 1 gives r = bf16(residual + x)."""
    B, S, D = 1, 5, 24
    i = _block(B, S, D, 4)
    one = np.full((B, D), 0x3F80, np.uint16)
    r0, _, _, _ = orc.res_fwd(i["x"], i["residual"], np.zeros((B, D), np.uint16), i["emb"])
    assert_bitwise(r0, i["residual"], "gate 0")
    r1, _, _, _ = orc.res_fwd(i["x"], np.zeros_like(i["x"]), i["gate"], i["emb"])
    assert_bitwise(r1, _bits_of(_tbf16(i["gate"])[:, None, :] * _tbf16(i["x"])), "residual 0")
    r2, _, _, _ = orc.res_fwd(i["x"], i["residual"], one, i["emb"])
    assert_bitwise(r2, _bits_of(_tbf16(i["residual"]) + _tbf16(i["x"])), "gate 1")


def test_res_bwd_tail_matches_torch_autograd_in_bf16(orc):
    """d_residual, d_x: the bf16 autograd of r = residual + gate * x (PyTorch
    on the CPU, bf16 tensors) given the gradient of r as the bf16 sum of its
    two uses; d_gate: the exact sum over tokens of the bf16 products gr * x
    (math.fsum), rounded once to fp32."""
    B, S, D = 2, 9, 32
    i = _block(B, S, D, 5)
    dr_ln = i["dy"]
    d_x, d_res, d_gate = orc.res_bwd_tail(dr_ln, i["dr"], i["x"], i["gate"])
    x = _tbf16(i["x"]).clone().requires_grad_(True)
    res = _tbf16(i["residual"]).clone().requires_grad_(True)
    gate = _tbf16(i["gate"])[:, None, :].clone().requires_grad_(True)
    r = res + gate * x
    gr = _tbf16(dr_ln) + _tbf16(i["dr"])
    r.backward(gr)
    assert_bitwise(d_res, _bits_of(res.grad), "d_residual")
    assert_bitwise(d_x, _bits_of(x.grad), "d_x")
    prod = bf16_to_f64(_bits_of(gr * _tbf16(i["x"])))
    want = np.array([[math.fsum(prod[b, :, d]) for d in range(D)] for b in range(B)]).astype(np.float32)
    assert_bitwise(d_gate, want, "d_gate")
    # without the later use, gr is dr_ln itself
    d_x0, d_res0, _ = orc.res_bwd_tail(dr_ln, None, i["x"], i["gate"])
    assert_bitwise(d_res0, dr_ln, "d_residual without d_r")
    assert_bitwise(d_x0, _bits_of(_tbf16(dr_ln) * _tbf16(i["gate"])[:, None, :]), "d_x without d_r")


def test_res_bwd_is_the_norm_backward_then_the_tail(orc):
    """The whole backward: d_emb and the LayerNorm input's gradient from the
    norm_out backward applied to r, then the tail; the gate products replayed
    by the fixed token tree stay within the tree's error bound of d_gate."""
    B, S, D = 2, 37, 24
    i = _block(B, S, D, 6)
    r, _, _, _ = orc.res_fwd(i["x"], i["residual"], i["gate"], i["emb"])
    d_x, d_res, d_emb, d_gate = orc.res_bwd(i["dy"], i["dr"], i["x"], r, i["gate"], i["emb"])
    dr_ln, w_demb = orc.out_bwd(i["dy"], r, i["emb"])
    assert_bitwise(d_emb, w_demb, "d_emb")
    w_dx, w_dres, w_dgate = orc.res_bwd_tail(dr_ln, i["dr"], i["x"], i["gate"])
    assert_bitwise(d_x, w_dx, "d_x")
    assert_bitwise(d_res, w_dres, "d_residual")
    assert_bitwise(d_gate, w_dgate, "d_gate")
    prod = orc.res_gate_products_f32(d_res, i["x"])
    assert_bitwise(prod, bf16_to_f64(_bits_of(_tbf16(d_res) * _tbf16(i["x"]))).astype(np.float32), "products")
    tree = orc.token_tree_f32(prod)
    exact = np.array([[math.fsum(prod[b, :, d].astype(np.float64)) for d in range(D)] for b in range(B)])
    bound = 2.0 ** -23 * np.abs(exact) + 2.0 ** -30 * np.abs(prod).astype(np.float64).sum(axis=1)
    assert np.all(np.abs(tree - exact) <= bound + 2.0 ** -24 * np.abs(exact))
    assert np.all(np.abs(d_gate.astype(np.float64) - exact) <= 2.0 ** -24 * np.abs(exact))


# ---------------------------------------------------------------------------
# fp32 execution dtype (RL-Kernel PR 538 "Results": the FP32 timings and gates)
# ---------------------------------------------------------------------------

def _f32_inputs(B, S, D, seed):
    rng = np.random.default_rng(seed)
    return {"x": rng.standard_normal((B, S, D)).astype(np.float32),
            "dy": rng.standard_normal((B, S, D)).astype(np.float32),
            "temb": rng.standard_normal((B, D)).astype(np.float32),
            "W": (rng.standard_normal((2 * D, D)) * 0.02).astype(np.float32),
            "b": (rng.standard_normal(2 * D) * 0.02).astype(np.float32)}


def _ulp32(a, b):
    ia = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    ib = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    ia = np.where(ia < 0, -(ia & 0x7FFFFFFF), ia)
    ib = np.where(ib < 0, -(ib & 0x7FFFFFFF), ib)
    return np.abs(ia - ib)


def test_f32_proj_fwd_exact(orc):
    """u = the fp32 nearest to silu(t) (mpmath at 200 bits); emb = the exact
    rational sum of u W + bias rounded once to fp32, bit for bit."""
    import mpmath
    mpmath.mp.prec = 200
    B, D = 2, 8
    i = _f32_inputs(B, 1, D, 40)
    emb, u = orc.f32_proj_fwd(i["temb"], i["W"], i["b"])
    for b in range(B):
        for k in range(D):
            t = mpmath.mpf(float(i["temb"][b, k]))
            s = t / (1 + mpmath.exp(-t))
            mag = Fraction(int(s.man)) * Fraction(2) ** int(s.exp)
            assert Fraction(float(u[b, k])) == f32_exact_round(-mag if s < 0 else mag), (b, k)
    for b in range(B):
        for n in range(2 * D):
            v = sum(Fraction(float(u[b, k])) * Fraction(float(i["W"][n, k])) for k in range(D))
            v += Fraction(float(i["b"][n]))
            assert Fraction(float(emb[b, n])) == f32_exact_round(v), (b, n)


def test_f32_out_fwd_rounding_points(orc):
    """out = fp32(fp32(xhat * fp32(1 + scale)) + shift) with xhat the fp32 of
    numpy's fp64 LayerNorm; the fused form and an unrounded (1 + scale) each
    give different bits somewhere, so neither could pass."""
    B, S, D = 2, 6, 64
    i = _f32_inputs(B, S, D, 41)
    emb = (np.random.default_rng(42).standard_normal((B, 2 * D)) * 0.3).astype(np.float32)
    out, mean, rstd = orc.f32_out_fwd(i["x"], emb)
    x = i["x"].astype(np.float64)
    mu = x.mean(-1, keepdims=True)
    var = ((x - mu) ** 2).mean(-1, keepdims=True)
    r = 1.0 / np.sqrt(var + EPS32)
    xh = ((x - mu) * r).astype(np.float32)
    onep = (np.float32(1) + emb[:, None, :D]).astype(np.float32)
    shift = emb[:, None, D:]
    want = (xh * onep).astype(np.float32) + shift
    assert np.all(_ulp32(out, want) <= 1) and (out == want).mean() > 0.999
    assert np.all(_ulp32(mean, mu[..., 0].astype(np.float32)) <= 1)
    assert np.all(_ulp32(rstd, r[..., 0].astype(np.float32)) <= 1)
    fused = (xh.astype(np.float64) * onep + shift).astype(np.float32)
    raw_onep = ((xh.astype(np.float64) * (1.0 + emb[:, None, :D].astype(np.float64))).astype(np.float32) + shift)
    assert np.any(fused != out) and np.any(raw_onep != out)


def test_f32_out_bwd_matches_torch_autograd(orc):
    """dx: torch fp64 autograd of xhat * onep (onep = fp32(1 + scale)) rounded
    to fp32, within 1 ulp; d_scale, d_shift: math.fsum of g * fp32(xhat) and of
    g, rounded once, bit for bit."""
    B, S, D = 2, 7, 48
    i = _f32_inputs(B, S, D, 43)
    emb = (np.random.default_rng(44).standard_normal((B, 2 * D)) * 0.3).astype(np.float32)
    dx, d_emb = orc.f32_out_bwd(i["dy"], i["x"], emb)
    x = torch.tensor(i["x"], dtype=torch.float64, requires_grad=True)
    onep = torch.tensor((np.float32(1) + emb[:, :D]).astype(np.float64))[:, None, :]
    y = torch.nn.functional.layer_norm(x, (D,), eps=EPS32) * onep
    y.backward(torch.tensor(i["dy"], dtype=torch.float64))
    want = x.grad.numpy().astype(np.float32)
    assert np.all(_ulp32(dx, want) <= 1) and (dx == want).mean() > 0.99
    xd = i["x"].astype(np.float64)
    mu = xd.mean(-1, keepdims=True)
    xh = ((xd - mu) / np.sqrt(((xd - mu) ** 2).mean(-1, keepdims=True) + EPS32)).astype(np.float32)
    g = i["dy"].astype(np.float64)
    for b in range(B):
        for d in range(D):
            assert d_emb[b, d] == np.float32(math.fsum(g[b, :, d] * xh[b, :, d].astype(np.float64)))
            assert d_emb[b, D + d] == np.float32(math.fsum(g[b, :, d]))


def test_f32_bwd_products_are_numpy_fp32_ops(orc):
    B, S, D = 2, 5, 32
    i = _f32_inputs(B, S, D, 45)
    rng = np.random.default_rng(46)
    mean = (rng.standard_normal((B, S)) * 2).astype(np.float32)
    rstd = np.exp(rng.uniform(-3, 3, (B, S))).astype(np.float32)
    prod = orc.f32_bwd_products(i["dy"], i["x"], mean, rstd)
    xh = ((i["x"] - mean[..., None]).astype(np.float32) * rstd[..., None]).astype(np.float32)
    assert_bitwise(prod[..., :D], (i["dy"] * xh).astype(np.float32), "g * xhat")
    assert_bitwise(prod[..., D:], i["dy"], "g")


def test_f32_proj_bwd_matches_torch_autograd(orc):
    """d_temb, dW, db: torch fp64 autograd of emb = fp32(silu(t)) @ W^T + b
    (the fp32 u treated as exact, silu' of t analytic), rounded to fp32."""
    B, D = 3, 16
    i = _f32_inputs(B, 1, D, 47)
    d_emb = np.random.default_rng(48).standard_normal((B, 2 * D)).astype(np.float32)
    d_temb, dW, db = orc.f32_proj_bwd(d_emb, i["temb"], i["W"])
    t = torch.tensor(i["temb"], dtype=torch.float64, requires_grad=True)
    s = torch.sigmoid(t)
    u32 = torch.tensor(orc.f32_proj_fwd(i["temb"], i["W"], i["b"])[1], dtype=torch.float64)
    u = u32 + (t * s - (t * s).detach())  # value fp32(silu(t)), gradient silu'(t)
    W = torch.tensor(i["W"], dtype=torch.float64, requires_grad=True)
    bb = torch.tensor(i["b"], dtype=torch.float64, requires_grad=True)
    (u @ W.T + bb).backward(torch.tensor(d_emb, dtype=torch.float64))
    assert np.all(_ulp32(d_temb, t.grad.numpy().astype(np.float32)) <= 1)
    assert np.all(_ulp32(dW, W.grad.numpy().astype(np.float32)) <= 1)
    assert np.all(_ulp32(db, bb.grad.numpy().astype(np.float32)) <= 1)


def test_f32_wgrad_seq_is_a_sequential_fused_multiply_add(orc):
    """acc = fp32(e * u + acc) (one rounding) over samples in ascending order,
    against exact rationals; a separately rounded product would differ."""
    B, D = 5, 6
    rng = np.random.default_rng(49)
    e = rng.standard_normal((B, 2 * D)).astype(np.float32)
    u = rng.standard_normal((B, D)).astype(np.float32)
    dW, db = orc.f32_wgrad_seq(e, u)
    unfused = 0
    for n in range(2 * D):
        for k in range(D):
            a = Fraction(0)
            a2 = np.float32(0)
            for b in range(B):
                a = f32_exact_round(Fraction(float(e[b, n])) * Fraction(float(u[b, k])) + a)
                a2 = np.float32(a2 + np.float32(e[b, n] * u[b, k]))
            assert Fraction(float(dW[n, k])) == a, (n, k)
            unfused += float(a2) != float(a)
    assert unfused > 0
    db_want = np.zeros(2 * D, np.float32)
    for b in range(B):
        db_want = (db_want + e[b]).astype(np.float32)
    assert_bitwise(db, db_want, "db")
    # accumulate: continuing from the accumulators equals one longer sequence
    dW1, db1 = orc.f32_wgrad_seq(e[:2], u[:2])
    dW2, db2 = orc.f32_wgrad_seq(e[2:], u[2:], dW1, db1, accumulate=True)
    assert_bitwise(dW2, dW, "chunked dW")
    assert_bitwise(db2, db, "chunked db")


# ---------------------------------------------------------------------------
# proj_out (RL-Kernel PR 538 "What": the latent projection 3072 -> 64)
# ---------------------------------------------------------------------------

def test_proj_out_exact_rational_and_torch(orc):
    """y = bf16(out Wp^T + bp): exact rational sums rounded once (bit for bit)
    on a small case; the fp64 map against torch.nn.functional.linear; Wp = 0
    gives y = bp; Wp's rows are the output features (a transposed Wp fails)."""
    rng = np.random.default_rng(50)
    R, D, J = 5, 16, 8
    out = _bf16(rng.standard_normal((R, D)))
    Wp = _bf16(rng.standard_normal((J, D)) * 0.1)
    bp = _bf16(rng.standard_normal(J) * 0.1)
    y = orc.proj_out(out, Wp, bp)
    of, wf, bf = bf16_to_f64(out), bf16_to_f64(Wp), bf16_to_f64(bp)
    for r in range(R):
        for j in range(J):
            v = sum(Fraction(float(of[r, d])) * Fraction(float(wf[j, d])) for d in range(D)) + Fraction(float(bf[j]))
            assert int(y[r, j]) == bf16_exact_round(v), (r, j)
    t = torch.nn.functional.linear(torch.tensor(of), torch.tensor(wf), torch.tensor(bf)).numpy()
    assert np.all(bf16_ulp_dist(y, orc.bf16_from_f64(t)) <= 1)
    assert_bitwise(orc.proj_out(out, np.zeros_like(Wp), bp), np.broadcast_to(bp, (R, J)).astype(np.uint16), "Wp = 0")
    sq = _bf16(rng.standard_normal((D, D)) * 0.1)
    assert not np.array_equal(orc.proj_out(out, sq, bp[:1].repeat(D)), orc.proj_out(out, sq.T.copy(), bp[:1].repeat(D)))
