"""The unscaled-cache ablation -- TEST INFRASTRUCTURE ONLY.

sgl-project/sglang-jax #1776, "feat(dsa): implement fp8 KV cache (e4m3) with a
bf16 indexer cache", design points and accuracy tests: the latent cache there
is cast to e4m3 or e5m2 with no scale at all (its values are O(1), post-
LayerNorm; fp8 precision is relative, so a power-of-two rescale would change
nothing), e4m3 is preferred for its extra mantissa bit (worst-case relative
rounding error about 6 % against about 12.5 % for e5m2), and, measured as the
attention error relative to the same cache kept in bf16, e5m2 does about twice
as badly as e4m3 (ratios 1.87-2.10 on that page).

This module states the caches the ablation compares and the attention it runs
on them, in float64, in the plainest form:

  bf16      the bf16 rows themselves (the reference cache);
  e4m3      each bf16 value cast to e4m3, no scale (round to nearest even,
            saturating at 448);
  e5m2      each bf16 value cast to e5m2, no scale (round to nearest even,
            saturating at 57344);
  e4m3_row  this library's cache: one fp32 scale per row (amax / 448), codes
            e4m3(x / scale) -- ROCm/ATOM PR #2655, PR description, K/V bullet.

The codecs are the C oracle's (oracle/kvq_oracle.c); the attention is a
textbook softmax attention (one matrix product, a max-subtracted softmax, a
second matrix product) with the multi-row causal rule of the paged oracle.
"""
from __future__ import annotations

import numpy as np

from . import (e4m3_decode, e4m3_encode, e5m2_decode, e5m2_encode, quantize_rows)

FORMATS = ("bf16", "e4m3", "e5m2", "e4m3_row")


def bf16_values(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 values (the upper half of a binary32)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def cache_values(fmt: str, x_bits: np.ndarray) -> np.ndarray:
    """The values a cache of format `fmt` holds for bf16 rows `x_bits`
    [..., D] (uint16 bit patterns), as float64 [..., D]."""
    x = bf16_values(x_bits)
    if fmt == "bf16":
        return x
    if fmt == "e4m3":
        return e4m3_decode(e4m3_encode(x.astype(np.float32)))
    if fmt == "e5m2":
        return e5m2_decode(e5m2_encode(x.astype(np.float32)))
    if fmt == "e4m3_row":
        codes, scales = quantize_rows(x_bits)
        return e4m3_decode(codes) * scales.astype(np.float64)[..., None]
    raise ValueError(fmt)


def attention_fp64(q: np.ndarray, K: np.ndarray, V: np.ndarray, sm_scale: float) -> np.ndarray:
    """Softmax attention of one request in float64.

    q [R, Hq, D] (the request's R query rows), K and V [L, H, D] (its cached
    tokens, the R newest last); GQA head hq reads KV head hq // (Hq // H); row
    i sees the first L - R + 1 + i tokens, a row that sees none gives zeros.
    Returns [R, Hq, D]."""
    R, Hq, D = q.shape
    L, H, _ = K.shape
    G = Hq // H
    out = np.zeros((R, Hq, D), dtype=np.float64)
    for i in range(R):
        vis = L - R + 1 + i
        if vis <= 0:
            continue
        for hq in range(Hq):
            h = hq // G
            s = sm_scale * (K[:vis, h, :] @ q[i, hq])            # [vis]
            p = np.exp(s - s.max())
            out[i, hq] = (p @ V[:vis, h, :]) / p.sum()
    return out


def rel_l2(got: np.ndarray, ref: np.ndarray) -> float:
    return float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
