"""Seeded synthetic inputs for the AdaLN ``norm_out`` operator.

This module only draws numbers.  It holds none of the operator's arithmetic,
so both sides of every parity check (the CUDA library and the CPU oracle)
can take their inputs from it without sharing any computation.

Generator (counter based, so any slice can be drawn on its own):

* ``splitmix64``: the 64-bit finaliser of Steele, Lea and Flood's SplitMix
  (constants 0x9E3779B97F4A7C15, 0xBF58476D1CE4E5B9, 0x94D049BB133111EB,
  shifts 30/27/31).  Element ``i`` of a stream with key ``k`` is
  ``mix(k + (i + 1) * 0x9E3779B97F4A7C15)``.
* Box-Muller in float64 on pairs of draws (53-bit uniforms), giving N(0, 1).
* ``value = mean + std * z`` in float64, rounded to float32, then rounded to
  bfloat16 with round-to-nearest-even.

Stream keys depend on (seed, tensor, sample), never on the batch size, so
sample ``b`` of a batch is bit-identical to the same sample drawn alone.
That is what the batch-invariance checks rely on.

Workload shapes follow the pages (RL-Kernel PR 538 "final_adaln_out",
section "What"): hidden size D = 3072, projection 3072 -> 6144, token
activations ``x``/``dy`` of shape [B, S, D], conditioning ``temb`` [B, D].
The real ``norm_out.linear`` weights the pages used are not available;
W and b are drawn from N(0, 0.02^2) instead.
"""

from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Tensor identifiers folded into the stream keys.
TENSOR_IDS = {"x": 1, "temb": 2, "W": 3, "b": 4, "dy": 5, "outlier": 6, "aux": 7, "residual": 8, "gate": 9,
              "emb": 10, "dr": 11}


def _mix(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64, copy=True)
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def stream_key(seed: int, tensor: str, sample: int = 0) -> int:
    """64-bit key of one stream, a function of (seed, tensor, sample) only."""
    tid = TENSOR_IDS[tensor]
    raw = np.array(
        [(seed & 0xFFFFFFFF) << 32 | (tid & 0xFF) << 24 | (sample & 0xFFFFFF)],
        dtype=np.uint64,
    )
    return int(_mix(raw)[0])


def splitmix64(key: int, start: int, n: int) -> np.ndarray:
    """Draws ``start .. start+n-1`` of the stream with the given key."""
    with np.errstate(over="ignore"):
        idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        return _mix(np.uint64(key) + idx * _GOLDEN)


def normal(key: int, n: int, start: int = 0) -> np.ndarray:
    """``n`` standard normals (float64) from element ``start`` of a stream.

    Normal ``j`` comes from the pair of draws (2*(j//2), 2*(j//2)+1): the
    cosine branch for even ``j``, the sine branch for odd ``j``.
    """
    if n == 0:
        return np.zeros(0, dtype=np.float64)
    p0 = start // 2
    p1 = (start + n + 1) // 2
    raw = splitmix64(key, 2 * p0, 2 * (p1 - p0)).reshape(-1, 2)
    scale = 1.0 / 9007199254740992.0  # 2^-53
    u1 = ((raw[:, 0] >> np.uint64(11)).astype(np.float64) + 1.0) * scale  # (0, 1]
    u2 = (raw[:, 1] >> np.uint64(11)).astype(np.float64) * scale  # [0, 1)
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * (p1 - p0), dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    off = start - 2 * p0
    return z[off:off + n]


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits.

    Inputs are finite.  NaN is kept a quiet NaN.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    out = rounded.astype(np.uint16)
    nan = (u & np.uint64(0x7FFFFFFF)) > np.uint64(0x7F800000)
    if nan.any():
        out[nan] = ((u[nan] >> np.uint64(16)) | np.uint64(0x40)).astype(np.uint16)
    return out


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bits to float32."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(key: int, n: int, std: float = 1.0, start: int = 0) -> np.ndarray:
    z = normal(key, n, start) * std
    return bf16_bits_from_f32(z.astype(np.float32))


def outlier_rows(seed: int, B: int, S: int, frac: float = 0.01) -> np.ndarray:
    """Flat row indices (b*S + s) of the outlier rows: floor(frac*B*S) rows,
    chosen by the seed without replacement, sorted ascending."""
    k = int(np.floor(frac * B * S))
    if k == 0:
        return np.zeros(0, dtype=np.int64)
    keys = splitmix64(stream_key(seed, "outlier"), 0, B * S)
    return np.sort(np.argsort(keys, kind="stable")[:k]).astype(np.int64)


def token_tensor(seed: int, tensor: str, B: int, S: int, D: int, sample0: int = 0,
                 outliers: np.ndarray | None = None, outlier_scale: float = 50.0) -> np.ndarray:
    """[B, S, D] bfloat16 bits of N(0, 1) tokens; rows listed in ``outliers``
    (flat b*S+s indices into this batch) are scaled in float32 by
    ``outlier_scale`` before the bfloat16 rounding."""
    out = np.empty((B, S, D), dtype=np.uint16)
    for b in range(B):
        z = normal(stream_key(seed, tensor, sample0 + b), S * D).astype(np.float32).reshape(S, D)
        if outliers is not None and len(outliers):
            rows = outliers[(outliers >= b * S) & (outliers < (b + 1) * S)] - b * S
            if len(rows):
                z[rows] = z[rows] * np.float32(outlier_scale)
        out[b] = bf16_bits_from_f32(z)
    return out


def make_inputs(B: int, S: int, D: int = 3072, seed: int = 0, sample0: int = 0,
                outlier_frac: float = 0.0, w_std: float = 0.02) -> dict:
    """All inputs of one forward+backward of the operator, as bfloat16 bits.

    x, dy: [B, S, D] ~ N(0, 1); temb: [B, D] ~ N(0, 1);
    W: [2D, D] ~ N(0, w_std^2) (row n = output feature n, (scale, shift) order);
    b: [2D] ~ N(0, w_std^2).
    With ``outlier_frac`` > 0, floor(frac*B*S) rows (the same rows in x and
    dy) are scaled by 50 in float32 before rounding.
    """
    rows = outlier_rows(seed, B, S, outlier_frac) if outlier_frac > 0 else None
    temb = np.stack([normal_bf16(stream_key(seed, "temb", sample0 + b), D) for b in range(B)]) \
        if B > 0 else np.zeros((0, D), dtype=np.uint16)
    return {
        "x": token_tensor(seed, "x", B, S, D, sample0, rows),
        "dy": token_tensor(seed, "dy", B, S, D, sample0, rows),
        "temb": temb.reshape(B, D),
        "W": normal_bf16(stream_key(seed, "W"), 2 * D * D, std=w_std).reshape(2 * D, D),
        "b": normal_bf16(stream_key(seed, "b"), 2 * D, std=w_std),
        "outlier_rows": rows if rows is not None else np.zeros(0, dtype=np.int64),
    }


def make_block_inputs(B: int, S: int, D: int = 3072, seed: int = 0, sample0: int = 0,
                      outlier_frac: float = 0.0) -> dict:
    """Inputs of the block-level modulated norm with a gated residual, as
    bfloat16 bits: x (the branch output), residual and dy (the gradient of the
    norm's output) [B, S, D] ~ N(0, 1), dr (the residual output's gradient
    from later uses) [B, S, D] ~ N(0, 1); gate [B, D] ~ N(0, 0.5^2) and emb =
    [scale | shift] [B, 2D] ~ N(0, 0.3^2), drawn per sample like temb.  The
    same outlier rows (x50) in x, residual, dy and dr."""
    rows = outlier_rows(seed, B, S, outlier_frac) if outlier_frac > 0 else None

    def per_sample(tensor, n, std):
        if B == 0:
            return np.zeros((0, n), dtype=np.uint16)
        return np.stack([normal_bf16(stream_key(seed, tensor, sample0 + b), n, std=std) for b in range(B)])

    return {
        "x": token_tensor(seed, "x", B, S, D, sample0, rows),
        "residual": token_tensor(seed, "residual", B, S, D, sample0, rows),
        "dy": token_tensor(seed, "dy", B, S, D, sample0, rows),
        "dr": token_tensor(seed, "dr", B, S, D, sample0, rows),
        "gate": per_sample("gate", D, 0.5).reshape(B, D),
        "emb": per_sample("emb", 2 * D, 0.3).reshape(B, 2 * D),
        "outlier_rows": rows if rows is not None else np.zeros(0, dtype=np.int64),
    }


def uniform_f32(key: int, n: int, lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    """``n`` float32 values uniform in [lo, hi) (for the standalone token tree)."""
    raw = splitmix64(key, 0, n)
    u = (raw >> np.uint64(11)).astype(np.float64) / 9007199254740992.0
    return (lo + (hi - lo) * u).astype(np.float32)
