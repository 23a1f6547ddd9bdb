"""Closed-form sizes of a KV cache and of a paged block pool.

Test infrastructure only (see the package docstring).

Every function here is the plain arithmetic the pages state; there is nothing
to approximate.
"""

from __future__ import annotations

import math


def kv_bytes(layers: int, heads: int, head_dim: int, seq_len: int, batch: int,
             bytes_per_elem: int) -> int:
    """KV-cache bytes = 2 (K and V) * L * H * d_head * s * B * bytes_dtype.

    [A] §2 (the KV-bytes formula, with L=28, H=8, d=128, B=4, s=8000 as its
    example); the same formula in [B] §3.1 and [C] §4.
    """
    return 2 * layers * heads * head_dim * seq_len * batch * bytes_per_elem


def kv_bytes_per_token(layers: int, heads: int, head_dim: int, bytes_per_elem: int) -> int:
    """Per-token KV footprint: the KV-bytes formula at s = B = 1 ([B] §3.1)."""
    return kv_bytes(layers, heads, head_dim, 1, 1, bytes_per_elem)


def blocks_needed(num_tokens: int, block_size: int) -> int:
    """Number of fixed-size blocks that hold ``num_tokens`` tokens: ceil(l / bs).

    [A] §1.2: a 600-token sequence in 16-token blocks takes ceil(600/16) = 38.
    """
    if num_tokens < 0 or block_size <= 0:
        raise ValueError("num_tokens must be >= 0 and block_size > 0")
    return -(-num_tokens // block_size)


def paged_tail_waste(num_tokens: int, block_size: int) -> int:
    """Slots allocated but unused: only the last, partly-filled block wastes space.

    [A] §1.2 states the bound waste < block_size; [E] §4.3 names the same
    internal fragmentation of the tail block.
    """
    return blocks_needed(num_tokens, block_size) * block_size - num_tokens


def fixed_bucket_waste_fraction(num_tokens: int, buckets=(128, 256, 512, 1024)) -> float:
    """Fraction of a fixed-length bucket left empty when the smallest bucket
    that fits ``num_tokens`` is chosen ([A] §1.1: 600 tokens in a 1024 bucket
    leaves more than 40% padding)."""
    fits = [b for b in sorted(buckets) if b >= num_tokens]
    if not fits:
        raise ValueError("no bucket is large enough")
    return (fits[0] - num_tokens) / fits[0]


def max_concurrent_requests(gpu_mem_bytes: float, mem_utilisation: float,
                            weight_bytes: float, kv_bytes_per_token_: float,
                            max_model_len: int) -> int:
    """Safe concurrency = floor((mem * utilisation - weights) / (per-token KV * max_len)).

    [B] §3.5: an 80 GB A100 at 0.9 utilisation with 14 GB of weights leaves
    58 GB; a 4096-token request needs 2 GB; about 29 requests fit.
    """
    available = gpu_mem_bytes * mem_utilisation - weight_bytes
    per_request = kv_bytes_per_token_ * max_model_len
    return int(math.floor(available / per_request))
