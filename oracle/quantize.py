"""Symmetric INT8 quantization of one KV block, and its dequantization.

Test infrastructure only (see the package docstring).

Source: [E] "轻量级推理引擎实战：KV Cache 量化与连续批处理的底层优化" §3, the
KV-cache quantizer: per head, take the largest absolute value, set the scale to
that maximum over 127 (1.0 when the head is all zero), quantize each value to
the nearest integer of x / scale clamped to [-127, 127], and dequantize with a
single multiply q * scale.

Readings (listed in the design notes):

* granularity: one scale per (block, kv_head, K|V) -- the maximum runs over
  the block's block_size x head_dim values of that head;
* the zero guard: scale = 1.0 when max|x| < 1e-6 (the page's comparison
  operator is lost in extraction; its comment says all-zero -> 1.0);
* rounding: fp32 IEEE division x / scale, then round-half-to-even
  (``rint``), then clamp -- rather than the page's reciprocal multiply with
  ties away from zero;
* arithmetic is fp32 throughout (the page's values are f32), so the result
  is bit-exact and a GPU implementation must reproduce it byte for byte.
"""

from __future__ import annotations

import numpy as np

QMAX = 127
ZERO_GUARD = np.float32(1e-6)


def block_scale(x: np.ndarray) -> np.float32:
    """Scale of one (block, kv_head, K|V) slab: max|x| / 127, or 1.0 if max|x| < 1e-6."""
    x = np.asarray(x, dtype=np.float32)
    m = np.float32(np.max(np.abs(x))) if x.size else np.float32(0.0)
    if m < ZERO_GUARD:
        return np.float32(1.0)
    return np.float32(m / np.float32(QMAX))


def quantize_block(x: np.ndarray):
    """Quantize one slab of bf16-valued fp32 data.

    ``x`` holds the block_size x head_dim values of one kv head of K (or V)
    in one block. Returns ``(q, scale)`` with ``q`` int8 of x's shape and
    ``scale`` an fp32 scalar.
    """
    x = np.asarray(x, dtype=np.float32)
    s = block_scale(x)
    r = np.rint(x / s)                       # fp32 division, ties to even
    q = np.clip(r, -QMAX, QMAX).astype(np.int8)
    return q, s


def dequantize(q: np.ndarray, scale) -> np.ndarray:
    """x_hat = q * scale, evaluated in fp64 (the oracle's attention precision)."""
    return np.asarray(q, dtype=np.float64) * np.float64(np.float32(scale))
