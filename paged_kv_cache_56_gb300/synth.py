"""Seeded, counter-based synthetic inputs (q, K, V rows; head multipliers; traces).

This module generates inputs only: it contains none of the cache's
arithmetic. Every value is a pure function of (seed, tensor identity, element
index), computed with integer hashing, a table lookup and at most one IEEE
fp32 multiply followed by round-to-nearest-even to bf16 -- operations whose
results are bit-identical on the CPU and on a GPU. A test can therefore
generate the full workload on the device and regenerate any slice of it on the
host, without copying data back.

Distribution: a value ~N(0, 1) is the standard-normal quantile at
(u + 1/2) / 65536 for a 16-bit hash u (a 65536-level inverse-CDF
quantization of the normal, |x| <= 4.3). Per-head multipliers are uniform on
a 65536-point grid.
"""

from __future__ import annotations

import math
from statistics import NormalDist

import numpy as np
import torch

M31 = 0x7FFFFFFF
_C1 = 0x045D9F3B
_C2 = 0x02B5A4ED
_SALT = 0x1F3D5B79

KIND_K, KIND_V, KIND_Q, KIND_MULT, KIND_OUTLIER, KIND_PERM = 0, 1, 2, 3, 4, 5


def _mix31(x: torch.Tensor) -> torch.Tensor:
    """31-bit multiply / fold hash. x: int64 tensor with values in [0, 2^31)."""
    x = x * _C1                                  # < 2^58, no int64 overflow
    x = (x ^ (x >> 31)) & M31
    x = x * _C2
    x = (x ^ (x >> 29)) & M31
    x = x * _C1
    x = (x ^ (x >> 31)) & M31
    return x


def _fold(h: torch.Tensor, x) -> torch.Tensor:
    """Fold a non-negative int64 (< 2^62) into the running hash h."""
    x = torch.as_tensor(x, dtype=torch.int64, device=h.device)
    h = _mix31(h ^ (x & M31))
    hi = (x >> 31) & M31
    return _mix31(h ^ hi ^ _SALT)


def row_key(seed: int, *ids, device="cpu") -> torch.Tensor:
    """Hash of (seed, ids...) -- ids may be ints or int64 tensors (broadcast)."""
    h = torch.tensor(seed & M31, dtype=torch.int64, device=device)
    for x in ids:
        h = _fold(h, x)
    return h


_NORM_TABLE_CPU = None
_NORM_TABLE_DEV = {}


def _norm_table(device) -> torch.Tensor:
    global _NORM_TABLE_CPU
    if _NORM_TABLE_CPU is None:
        nd = NormalDist()
        vals = [nd.inv_cdf((i + 0.5) / 65536.0) for i in range(65536)]
        _NORM_TABLE_CPU = torch.tensor(vals, dtype=torch.float64).to(torch.float32)
    dev = torch.device(device)
    if dev.type == "cpu":
        return _NORM_TABLE_CPU
    key = str(dev)
    if key not in _NORM_TABLE_DEV:
        _NORM_TABLE_DEV[key] = _NORM_TABLE_CPU.to(dev)
    return _NORM_TABLE_DEV[key]


def _u16(key: torch.Tensor, idx: torch.Tensor) -> torch.Tensor:
    h = _mix31(_mix31(key ^ (idx & M31)) ^ ((idx >> 31) & M31) ^ _SALT)
    return (h >> 7) & 0xFFFF


def normal_f32(key: torch.Tensor, idx: torch.Tensor) -> torch.Tensor:
    """N(0,1) fp32 values for element indices ``idx`` under stream ``key``."""
    return _norm_table(idx.device)[_u16(key, idx)]


def uniform_f32(key: torch.Tensor, idx: torch.Tensor, lo: float, hi: float) -> torch.Tensor:
    u = (_u16(key, idx).to(torch.float32) + 0.5) * (1.0 / 65536.0)
    return torch.tensor(lo, dtype=torch.float32, device=idx.device) + u * torch.tensor(
        hi - lo, dtype=torch.float32, device=idx.device)


# ---------------------------------------------------------------------------
# Workload-level generators
# ---------------------------------------------------------------------------

def head_multipliers(seed: int, layer: int, kind: int, n_heads: int, lo: float = 0.1,
                     hi: float = 4.0) -> torch.Tensor:
    """Per-head multipliers ~U(lo, hi), fixed per (layer, kind): fp32 [n_heads] (CPU)."""
    key = row_key(seed, KIND_MULT, layer, kind)
    return uniform_f32(key, torch.arange(n_heads, dtype=torch.int64), lo, hi)


def outlier_multipliers(seed: int, layer: int, kind: int, n_heads: int, head_dim: int,
                        prob: float = 0.01, factor: float = 20.0) -> torch.Tensor:
    """fp32 [n_heads, head_dim]: ``factor`` on a seeded ~prob fraction of dims, else 1."""
    key = row_key(seed, KIND_OUTLIER, layer, kind)
    u = uniform_f32(key, torch.arange(n_heads * head_dim, dtype=torch.int64), 0.0, 1.0)
    m = torch.where(u < prob, torch.tensor(factor, dtype=torch.float32),
                    torch.tensor(1.0, dtype=torch.float32))
    return m.reshape(n_heads, head_dim)


def _scaled_bf16(vals: torch.Tensor, mult) -> torch.Tensor:
    if mult is not None:
        vals = vals * mult.to(device=vals.device, dtype=torch.float32)
    return vals.to(torch.bfloat16)


def kv_rows(seed: int, layer: int, kind: int, seqs, positions, n_kv_heads: int,
            head_dim: int, mult=None, device="cpu", chunk_rows: int = 1 << 16) -> torch.Tensor:
    """K (kind=KIND_K) or V (KIND_V) rows of token ``positions[i]`` of sequence
    ``seqs[i]``: bf16 [T, n_kv_heads, head_dim].

    ``mult``: None, or fp32 broadcastable to [n_kv_heads, head_dim] (per-head
    scale, outlier channels). ``seqs`` may be an int (one sequence).
    """
    positions = torch.as_tensor(positions, dtype=torch.int64).to(device).reshape(-1)
    seqs = torch.as_tensor(seqs, dtype=torch.int64).to(device).reshape(-1)
    if seqs.numel() == 1 and positions.numel() != 1:
        seqs = seqs.expand(positions.numel())
    t = positions.numel()
    out = torch.empty((t, n_kv_heads, head_dim), dtype=torch.bfloat16, device=device)
    inner = torch.arange(n_kv_heads * head_dim, dtype=torch.int64, device=device)
    if mult is not None:
        mult = torch.as_tensor(mult, dtype=torch.float32).to(device)
        mult = mult.expand(n_kv_heads, head_dim) if mult.dim() == 2 else \
            mult.reshape(n_kv_heads, 1).expand(n_kv_heads, head_dim)
    for s in range(0, t, chunk_rows):
        e = min(t, s + chunk_rows)
        key = row_key(seed, kind, layer, seqs[s:e], device=device)[:, None]
        idx = positions[s:e, None] * (n_kv_heads * head_dim) + inner[None, :]
        vals = normal_f32(key, idx).reshape(e - s, n_kv_heads, head_dim)
        out[s:e] = _scaled_bf16(vals, mult)
    return out


def q_rows(seed: int, layer: int, step, seqs, n_q_heads: int, head_dim: int, mult=None,
           device="cpu") -> torch.Tensor:
    """Query rows of decode ``step`` for sequences ``seqs``: bf16 [B, Hq, d]."""
    seqs = torch.as_tensor(seqs, dtype=torch.int64).to(device).reshape(-1)
    step = torch.as_tensor(step, dtype=torch.int64).to(device).reshape(-1)
    if step.numel() == 1:
        step = step.expand(seqs.numel())
    key = row_key(seed, KIND_Q, layer, seqs, step, device=device)[:, None]
    idx = torch.arange(n_q_heads * head_dim, dtype=torch.int64, device=device)[None, :]
    vals = normal_f32(key, idx).reshape(-1, n_q_heads, head_dim)
    if mult is not None:
        mult = torch.as_tensor(mult, dtype=torch.float32).to(device)
        mult = mult.reshape(n_q_heads, 1) if mult.dim() == 1 else mult
    return _scaled_bf16(vals, mult)


def permutation(seed: int, n: int, salt: int = 0) -> list:
    """A seeded permutation of range(n) (argsort of hashes, ties by index)."""
    key = row_key(seed, KIND_PERM, salt)
    h = _mix31(key ^ torch.arange(n, dtype=torch.int64))
    order = sorted(range(n), key=lambda i: (int(h[i]), i))
    return order


# ---------------------------------------------------------------------------
# Continuous-batching trace (host control data only)
# ---------------------------------------------------------------------------

def trace_requests(seed: int, num_steps: int, arrival_rate: float = 2.0,
                   prompt_min: int = 16, prompt_max: int = 4096, mean_output: float = 300.0):
    """Arrivals for a continuous-batching trace.

    Returns a list of (arrival_step, request_id, prompt_len, output_len):
    Poisson(arrival_rate) arrivals per step, prompt length
    round(exp(U(ln min, ln max))), output length ~ Geometric(1/mean) >= 1.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    reqs = []
    rid = 0
    for step in range(num_steps):
        for _ in range(int(rng.poisson(arrival_rate))):
            p = int(round(math.exp(rng.uniform(math.log(prompt_min), math.log(prompt_max)))))
            p = min(max(p, prompt_min), prompt_max)
            o = int(rng.geometric(1.0 / mean_output))
            reqs.append((step, rid, p, max(o, 1)))
            rid += 1
    return reqs
