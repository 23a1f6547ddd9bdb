"""How many requests a KV memory budget holds under three ways of reserving
cache memory ("无 vLLM 环境下的 Paged-KV 与连续批处理调度" §1.1-1.2;
"vLLM核心概念" §3.5):

* ``bucket``: every request reserves the smallest of a fixed set of lengths
  that holds it (§1.1's compiled 128/256/512/1024... buckets) -- padding up
  to the bucket is internal fragmentation;
* ``max_len``: every request reserves the model's maximum length (§3.5's
  "safe concurrency" = budget / per-request maximum);
* ``paged``: ceil(length / block_size) blocks, waste below one block (§1.2);
* ``paged_int8``: the same blocks at one byte per element plus this cache's
  per-(block, kv head, K|V) fp32 scales and each running request's bf16 tail
  block (the partly filled block stays bf16 until it fills).

Host arithmetic only: it sizes pools and admission limits; nothing here
touches the device.
"""

from __future__ import annotations

from dataclasses import dataclass

BUCKETS = (128, 256, 512, 1024, 2048, 4096)


@dataclass(frozen=True)
class KVShape:
    layers: int
    kv_heads: int
    head_dim: int

    def bytes_per_token(self, elem_bytes: int) -> int:
        """2 (K and V) * layers * kv heads * head_dim * element bytes."""
        return 2 * self.layers * self.kv_heads * self.head_dim * elem_bytes


def reserved_bytes(length: int, scheme: str, shape: KVShape, block_size: int = 16,
                   buckets=BUCKETS, max_len: int = 4096) -> int:
    """Cache bytes one request of ``length`` tokens holds under ``scheme``
    (bf16 elements unless the scheme is paged_int8)."""
    if length < 0:
        raise ValueError("length must be >= 0")
    bf16_tok = shape.bytes_per_token(2)
    if scheme == "bucket":
        fits = [b for b in sorted(buckets) if b >= length]
        if not fits:
            raise ValueError(f"no bucket holds {length} tokens")
        return fits[0] * bf16_tok
    if scheme == "max_len":
        if length > max_len:
            raise ValueError(f"{length} tokens exceed max_len {max_len}")
        return max_len * bf16_tok
    nblocks = -(-length // block_size)
    if scheme == "paged":
        return nblocks * block_size * bf16_tok
    if scheme == "paged_int8":
        full = length // block_size
        scales = full * shape.layers * shape.kv_heads * 2 * 4
        tail = block_size * bf16_tok  # the slot's bf16 tail, held while the request runs
        return full * block_size * shape.bytes_per_token(1) + scales + tail
    raise ValueError(f"unknown scheme {scheme!r}")


def concurrency(lengths, budget_bytes: int, scheme: str, shape: KVShape, **kw) -> int:
    """Requests admitted in order until the next one no longer fits."""
    used, n = 0, 0
    for ell in lengths:
        need = reserved_bytes(int(ell), scheme, shape, **kw)
        if used + need > budget_bytes:
            break
        used += need
        n += 1
    return n


def waste_fraction(lengths, scheme: str, shape: KVShape, **kw) -> float:
    """Share of the reserved bytes that holds no token (bf16 accounting)."""
    held = sum(reserved_bytes(int(ell), scheme, shape, **kw) for ell in lengths)
    if scheme == "paged_int8":
        payload = sum(int(ell) * shape.bytes_per_token(1) for ell in lengths)
    else:
        payload = sum(int(ell) * shape.bytes_per_token(2) for ell in lengths)
    return 1.0 - payload / held if held else 0.0


def study(lengths, budget_bytes: int, shape: KVShape, block_size: int = 16, buckets=BUCKETS,
          max_len: int = 4096) -> dict:
    """Concurrency and waste of every scheme for one length mix and budget."""
    out = {}
    for scheme in ("max_len", "bucket", "paged", "paged_int8"):
        kw = dict(block_size=block_size, buckets=buckets, max_len=max_len)
        out[scheme] = dict(requests=concurrency(lengths, budget_bytes, scheme, shape, **kw),
                           waste=waste_fraction(lengths, scheme, shape, **kw))
    return out


def trace_lengths(seed: int, n: int, prompt_min: int = 16, prompt_max: int = 4096,
                  mean_output: float = 300.0, max_len: int = 4096) -> list:
    """Context lengths of n requests caught mid-generation: prompt
    log-uniform in [prompt_min, prompt_max], a uniform share of an output
    length drawn geometric with the given mean (the trace workload's mix),
    capped at max_len."""
    import numpy as np
    rng = np.random.default_rng(seed)
    prompt = np.round(np.exp(rng.uniform(np.log(prompt_min), np.log(prompt_max), n))).astype(int)
    out = rng.geometric(1.0 / mean_output, n)
    done = np.floor(rng.uniform(0, 1, n) * out).astype(int)
    return [int(x) for x in np.minimum(prompt + done, max_len)]


if __name__ == "__main__":
    shape = KVShape(layers=32, kv_heads=32, head_dim=128)  # the pages' 7B example: 512 KB/token
    budget = 58 * 2 ** 30                                  # their 80 GB x 0.9 - 14 GB
    lengths = trace_lengths(1234, 4000)
    for scheme, r in study(lengths, budget, shape).items():
        print(f"{scheme:11s} requests {r['requests']:5d}  waste {100 * r['waste']:5.1f}%")
