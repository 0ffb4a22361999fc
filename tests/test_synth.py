"""The seeded input generator: determinism, slicing, per-sample independence
from the batch size, distributions and the bf16 rounding of inputs."""

from __future__ import annotations

from fractions import Fraction

import numpy as np

from invariant_dit_adaln_gb300 import synth


def test_splitmix64_reference_values():
    # SplitMix64 with state 0: the first outputs of the published generator
    # (Steele, Lea, Flood; also the seeding generator of xoshiro).
    got = synth.splitmix64(0, 0, 3)
    assert [int(v) for v in got] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_streams_are_sliceable_and_deterministic():
    k = synth.stream_key(7, "x", 3)
    full = synth.normal(k, 1001)
    for a, b in [(0, 10), (1, 17), (500, 1001), (333, 334)]:
        np.testing.assert_array_equal(synth.normal(k, b - a, start=a), full[a:b])
    np.testing.assert_array_equal(synth.normal(k, 1001), full)


def test_sample_content_does_not_depend_on_batch():
    big = synth.make_inputs(B=5, S=3, D=64, seed=11)
    for b in range(5):
        one = synth.make_inputs(B=1, S=3, D=64, seed=11, sample0=b)
        np.testing.assert_array_equal(one["x"][0], big["x"][b])
        np.testing.assert_array_equal(one["dy"][0], big["dy"][b])
        np.testing.assert_array_equal(one["temb"][0], big["temb"][b])
        np.testing.assert_array_equal(one["W"], big["W"])


def test_distributions():
    inp = synth.make_inputs(B=2, S=64, D=256, seed=0)
    x = synth.bf16_bits_to_f32(inp["x"]).astype(np.float64)
    W = synth.bf16_bits_to_f32(inp["W"]).astype(np.float64)
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1) < 0.02
    assert abs(W.mean()) < 0.001 and abs(W.std() - 0.02) < 0.001
    assert not np.array_equal(inp["x"], inp["dy"])


def test_outlier_rows():
    B, S, D = 2, 4096, 32
    rows = synth.outlier_rows(0, B, S)
    assert len(rows) == 81 and len(np.unique(rows)) == 81
    inp = synth.make_inputs(B=B, S=S, D=D, seed=0, outlier_frac=0.01)
    np.testing.assert_array_equal(inp["outlier_rows"], rows)
    x = synth.bf16_bits_to_f32(inp["x"]).reshape(B * S, D).astype(np.float64)
    rms = np.sqrt((x ** 2).mean(1))
    mask = np.zeros(B * S, bool)
    mask[rows] = True
    assert rms[mask].min() > 20 and rms[~mask].max() < 3


def test_bf16_rounding_is_nearest_even():
    rng = np.random.default_rng(0)
    f = (rng.standard_normal(2000) * np.exp2(rng.integers(-30, 30, 2000))).astype(np.float32)
    ties = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 2.0 ** -130 * 1.5], np.float32)
    f = np.concatenate([f, ties])
    got = synth.bf16_bits_from_f32(f)
    for v, h in zip(f, got):
        fv = Fraction(float(v))
        cand = [int(h) - 1, int(h), int(h) + 1]
        dists = [abs(Fraction(float(synth.bf16_bits_to_f32(np.array([c & 0xFFFF], np.uint16))[0])) - fv) for c in cand]
        assert dists[1] <= min(dists)
        if dists[1] == min(dists[0], dists[2]):  # tie: even mantissa
            assert int(h) % 2 == 0
