"""Host checks of two equivalences the CUDA path relies on, in IEEE fp32 (numpy
float32 arithmetic rounds each operation to nearest even and never fuses):

- the Neumaier step of the token tree (RL-Kernel PR 538, review thread on the
  cancellation case) computed as Knuth's branch-free TwoSum gives the same
  (sum, correction) bits whenever the sum is finite;
- a level-0 tile that starts from (+0, +0) instead of from its first token
  ends with the same bits, except that a column of zeros may differ in the
  sign of its sum, and its root (sum + correction) is +0 either way.

Both forms are written here from their definitions, independently of the
oracle and of the kernels."""

from __future__ import annotations

import numpy as np

f32 = np.float32


def neumaier_step(s, c, v):
    t = s + v
    big = np.abs(s) >= np.abs(v)
    lost = np.where(big, (s - t) + v, (v - t) + s)
    return t, c + lost


def twosum_step(s, c, v):
    t = s + v
    bp = t - s
    e = (s - (t - bp)) + (v - bp)
    return t, c + e


def _values(rng, n):
    """fp32 values over a wide exponent range, with exact ties, signed zeros,
    subnormals and repeated magnitudes of both signs."""
    mant = rng.uniform(1.0, 2.0, n)
    expo = rng.integers(-140, 100, n)
    v = (mant * np.exp2(expo.astype(np.float64)) * rng.choice([-1.0, 1.0], n)).astype(f32)
    pick = rng.random(n)
    v[pick < 0.05] = f32(0.0)
    v[(pick >= 0.05) & (pick < 0.10)] = f32(-0.0)
    v[(pick >= 0.10) & (pick < 0.15)] = (rng.integers(-3, 4, int(((pick >= 0.10) & (pick < 0.15)).sum()))
                                         .astype(f32) * f32(2.0 ** -149))
    return v


def bits(a):
    return np.ascontiguousarray(a, dtype=f32).view(np.uint32)


def test_twosum_equals_neumaier_bitwise():
    rng = np.random.default_rng(17)
    with np.errstate(over="ignore", invalid="ignore"):
        for _ in range(20):
            n = 200_000
            s = _values(rng, n)
            c = _values(rng, n) * f32(2.0 ** -30)
            v = _values(rng, n)
            # exact ties |s| == |v| of both signs, and near-cancellations
            k = n // 10
            v[:k] = -s[:k]
            v[k:2 * k] = s[k:2 * k]
            v[2 * k:3 * k] = (-s[2 * k:3 * k] * f32(1.0 + 2.0 ** -20)).astype(f32)
            t1, c1 = neumaier_step(s, c, v)
            t2, c2 = twosum_step(s, c, v)
            fin = np.isfinite(t1)
            assert np.array_equal(bits(t1[fin]), bits(t2[fin]))
            assert np.array_equal(bits(c1[fin]), bits(c2[fin]))


def test_tree_start_from_zero_equals_start_from_first_token():
    rng = np.random.default_rng(18)
    lanes, T = 50_000, 32
    vals = np.stack([_values(rng, lanes) for _ in range(T)])
    vals[:, : lanes // 20] = f32(-0.0)                  # columns of zeros only
    vals[:, lanes // 20: lanes // 10] = f32(0.0)
    vals[: T // 2, lanes // 10: lanes // 5] = f32(-0.0)  # zeros, then values
    with np.errstate(over="ignore", invalid="ignore"):
        s_a, c_a = vals[0].copy(), np.zeros(lanes, f32)
        for i in range(1, T):
            s_a, c_a = neumaier_step(s_a, c_a, vals[i])
        s_b, c_b = np.zeros(lanes, f32), np.zeros(lanes, f32)
        for i in range(T):
            s_b, c_b = twosum_step(s_b, c_b, vals[i])
    fin = np.isfinite(s_a) & np.isfinite(s_b)
    zero_col = np.all(vals == 0, axis=0)
    same = fin & ~zero_col
    assert np.array_equal(bits(s_a[same]), bits(s_b[same]))
    assert np.array_equal(bits(c_a[same]), bits(c_b[same]))
    # columns of zeros: the sums may differ in sign only; the roots are +0 both
    root_a = s_a[zero_col] + c_a[zero_col]
    root_b = s_b[zero_col] + c_b[zero_col]
    assert np.all(s_a[zero_col] == 0) and np.all(s_b[zero_col] == 0)
    assert np.array_equal(bits(root_a), np.zeros(int(zero_col.sum()), np.uint32))
    assert np.array_equal(bits(root_b), np.zeros(int(zero_col.sum()), np.uint32))
