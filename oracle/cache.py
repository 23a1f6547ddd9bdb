"""Contiguous per-sequence KV histories: the cache a paged layout must equal.

Test infrastructure only (see the package docstring).

A ``SequenceHistory`` keeps one sequence's K and V rows of one layer in token
order, with no paging at all. In INT8 mode it quantizes each block of
``block_size`` tokens at the moment the block fills, per (kv_head, K|V), with
``quantize.quantize_block``; the tokens of a block that has not filled yet
stay at their bf16 values. ``context()`` returns what one decode step attends
over: dequantized full blocks followed by the raw tail.

Sources: blocks of block_size tokens and per-sequence block lists ([A] §1.2,
[E] §2.1); quantization per head with a scale per block ([E] §3). The reading
that a block is quantized once, when it fills, and that the partial tail
block stays bf16 is listed in the design notes; the page's own note
quantizes later, when a block leaves fast memory.
"""

from __future__ import annotations

import numpy as np

from .quantize import quantize_block, dequantize


class SequenceHistory:
    def __init__(self, num_kv_heads: int, head_dim: int, block_size: int, int8: bool):
        self.hkv = num_kv_heads
        self.d = head_dim
        self.bs = block_size
        self.int8 = int8
        self._k = np.zeros((0, num_kv_heads, head_dim), dtype=np.float32)
        self._v = np.zeros((0, num_kv_heads, head_dim), dtype=np.float32)
        self.n = 0
        # block index -> (qk [Hkv,bs,d] int8, sk [Hkv] f32, qv, sv)
        self.blocks = {}

    def _reserve(self, n_new: int) -> None:
        cap = self._k.shape[0]
        if n_new <= cap:
            return
        cap = max(n_new, 2 * cap, 64)
        for name in ("_k", "_v"):
            old = getattr(self, name)
            new = np.zeros((cap, self.hkv, self.d), dtype=np.float32)
            new[: self.n] = old[: self.n]
            setattr(self, name, new)

    def append(self, k_rows: np.ndarray, v_rows: np.ndarray) -> list:
        """Append T tokens (rows [T, Hkv, d] of bf16 values). Returns the indices
        of the blocks that filled (and, in INT8 mode, were quantized)."""
        k_rows = np.asarray(k_rows, dtype=np.float32).reshape(-1, self.hkv, self.d)
        v_rows = np.asarray(v_rows, dtype=np.float32).reshape(-1, self.hkv, self.d)
        t = k_rows.shape[0]
        self._reserve(self.n + t)
        self._k[self.n: self.n + t] = k_rows
        self._v[self.n: self.n + t] = v_rows
        first_full_before = self.n // self.bs
        self.n += t
        filled = list(range(first_full_before, self.n // self.bs))
        if self.int8:
            for i in filled:
                self.blocks[i] = self._quantize(i)
        return filled

    def _quantize(self, i: int):
        bs, d, hkv = self.bs, self.d, self.hkv
        sl = slice(i * bs, (i + 1) * bs)
        qk = np.empty((hkv, bs, d), dtype=np.int8)
        qv = np.empty((hkv, bs, d), dtype=np.int8)
        sk = np.empty(hkv, dtype=np.float32)
        sv = np.empty(hkv, dtype=np.float32)
        for h in range(hkv):
            qk[h], sk[h] = quantize_block(self._k[sl, h, :])
            qv[h], sv[h] = quantize_block(self._v[sl, h, :])
        return qk, sk, qv, sv

    @property
    def num_full_blocks(self) -> int:
        return self.n // self.bs

    def raw(self):
        """The bf16-valued rows as appended: [n, Hkv, d] float32 each."""
        return self._k[: self.n], self._v[: self.n]

    def context(self, kv_heads=None):
        """K_hat, V_hat [n, Hkv, d] fp64: what a decode step attends over."""
        k, v = self.raw()
        k = k.astype(np.float64)
        v = v.astype(np.float64)
        if self.int8:
            bs = self.bs
            for i in range(self.num_full_blocks):
                qk, sk, qv, sv = self.blocks[i]
                sl = slice(i * bs, (i + 1) * bs)
                for h in range(self.hkv):
                    k[sl, h, :] = dequantize(qk[h], sk[h])
                    v[sl, h, :] = dequantize(qv[h], sv[h])
        if kv_heads is not None:
            k = k[:, kv_heads, :]
            v = v[:, kv_heads, :]
        return k, v
