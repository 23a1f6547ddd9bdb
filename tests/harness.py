"""Test harness: one seeded workload driven through the C ABI (GPU) and,
independently, through the oracle (CPU), from the same counter-based inputs.

Nothing here computes cache arithmetic: the GPU side calls libpkv.so through
the runtime, the CPU side calls ``oracle``. Both read their inputs from
``paged_kv_cache_56_gb300.synth``, which regenerates any row on any device.
"""

from __future__ import annotations

import math

import numpy as np
import torch

from oracle.attention import decode_attention
from oracle.cache import SequenceHistory
from paged_kv_cache_56_gb300 import pkv, synth
from paged_kv_cache_56_gb300.runtime import (GraphStep, PagedKVCache, StepBuffers, decode_step,
                                              plan_split_tokens, prefill)

ATOL, RTOL = 2e-3, 1e-2  # |gpu - ref| <= ATOL + RTOL * |ref| on bf16 outputs


def assert_close(gpu: np.ndarray, ref: np.ndarray, what: str = "") -> None:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bad = np.abs(gpu - ref) > ATOL + RTOL * np.abs(ref)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first at {tuple(i)}: "
                             f"gpu {gpu[tuple(i)]!r} ref {ref[tuple(i)]!r}; max err "
                             f"{np.max(np.abs(gpu - ref)):.3g}")


class Workload:
    """L layers, B sequences with prior lengths ``prior``; decode steps t = 0, 1, ..."""

    def __init__(self, seed: int, num_layers: int, prior, Hq: int, Hkv: int, d: int, bs: int,
                 num_blocks: int, int8, split_tokens: int = 0, max_blocks: int | None = None,
                 head_scale: bool = False, outliers: bool = False, shuffle: bool = True,
                 req_ids=None, device="cuda", fused_merge: bool = True, graph: bool = False, repeat: int = 1,
                 fused_step: bool | None = None, kv_scale=None):
        """kv_scale: optional fn(layer, kind, positions) -> fp32 [T, Hkv] (CPU)
        multiplying the generated K (kind synth.KIND_K) or V rows of tokens at
        ``positions`` per kv head (applied in fp32, then rounded to bf16: the
        same bits on either device)."""
        self.seed, self.L, self.prior = seed, num_layers, list(prior)
        self.Hq, self.Hkv, self.d, self.bs = Hq, Hkv, d, bs
        self.int8 = int8
        self.head_scale, self.outliers = head_scale, outliers
        self.kv_scale = kv_scale
        self.B = len(self.prior)
        self.req_ids = list(req_ids) if req_ids is not None else list(range(100, 100 + self.B))
        self.sm_scale = 1.0 / math.sqrt(d)
        self.device = device
        self.max_blocks = max_blocks or -(-(max(self.prior) + 64) // bs)
        order = synth.permutation(seed, num_blocks) if shuffle else None
        self.cache = PagedKVCache(num_layers, num_blocks, Hq, Hkv, d, bs, int8, max_slots=self.B,
                                  max_blocks_per_seq=self.max_blocks, device=device, initial_order=order)
        if split_tokens == "auto":  # as the benchmark sizes it: one wave of CTAs
            split_tokens = plan_split_tokens(self.cache, self.B, self.max_blocks * bs)
        self.split_tokens = split_tokens
        self.bufs = StepBuffers(self.cache, self.B, split_tokens, fused_merge=fused_merge)
        self.step_no = 0
        self.graph = graph
        self.R = repeat
        self.gs = None
        # fused_step: one pkv_decode_step per layer (the benchmark's path);
        # default on for graph replay, off for the eager three-kernel path
        self.fused_step = graph if fused_step is None else fused_step
        # the benchmark's launch configuration uses programmatic dependent launch
        pkv.pkv_set_programmatic_launch(graph)
        for r, n in zip(self.req_ids, self.prior):
            self.cache.add_sequence(r, -(-n // bs))
        for li in range(num_layers):
            ks = [self.kv(li, synth.KIND_K, r, torch.arange(n)) for r, n in zip(self.req_ids, self.prior)]
            vs = [self.kv(li, synth.KIND_V, r, torch.arange(n)) for r, n in zip(self.req_ids, self.prior)]
            prefill(self.cache, li, self.req_ids, ks, vs)
        for r, n in zip(self.req_ids, self.prior):
            self.cache.seqs[r].length = n
        torch.cuda.synchronize()

    # -- inputs (shared generator) ------------------------------------------
    def kv_mult(self, layer, kind):
        if self.outliers:
            return synth.outlier_multipliers(self.seed, layer, kind, self.Hkv, self.d)
        if self.head_scale:
            return synth.head_multipliers(self.seed, layer, kind, self.Hkv)
        return None

    def q_mult(self, layer):
        return synth.head_multipliers(self.seed, layer, synth.KIND_Q, self.Hq) if self.head_scale else None

    def kv(self, layer, kind, req, positions, device=None):
        rows = synth.kv_rows(self.seed, layer, kind, req, positions, self.Hkv, self.d,
                             mult=self.kv_mult(layer, kind), device=device or self.device)
        if self.kv_scale is not None:
            pos = torch.as_tensor(positions, dtype=torch.int64).reshape(-1).cpu()
            m = self.kv_scale(layer, kind, pos).to(torch.float32).to(rows.device)
            rows = (rows.float() * m[:, :, None]).to(torch.bfloat16)
        return rows

    def q(self, layer, step, reqs, device=None):
        return synth.q_rows(self.seed, layer, step, reqs, self.Hq, self.d, mult=self.q_mult(layer),
                            device=device or self.device)

    # -- GPU ------------------------------------------------------------------
    def q_for(self, qi, step, reqs, device=None):
        """Query of attention call qi (= layer * R + repeat) at decode step ``step``.
        Repeat r > 0 of a layer draws its own query stream."""
        layer, rep = divmod(qi, self.R)
        if rep == 0:
            return self.q(layer, step, reqs, device)
        return synth.q_rows(self.seed, 1000 * (rep + 1) + layer, step, reqs, self.Hq, self.d,
                            mult=self.q_mult(layer), device=device or self.device)

    def step(self):
        """One decode step through the C ABI; returns out [L*R, B, Hq, d] (device bf16).
        With graph=True the step runs as the bench runs it: one eager step, then
        replays of the captured CUDA graph."""
        t = self.step_no
        lens = [self.cache.seqs[r].length for r in self.req_ids]
        pos = torch.tensor(lens, dtype=torch.int64)
        q = torch.stack([self.q_for(qi, t, self.req_ids) for qi in range(self.L * self.R)])
        kn = torch.stack([self.kv(li, synth.KIND_K, self.req_ids, pos) for li in range(self.L)])
        vn = torch.stack([self.kv(li, synth.KIND_V, self.req_ids, pos) for li in range(self.L)])
        if not self.graph and self.R == 1 and not self.fused_step:
            out = torch.empty((self.L, self.B, self.Hq, self.d), dtype=torch.bfloat16, device=self.device)
            decode_step(self.cache, self.bufs, self.req_ids, list(q), list(kn), list(vn), list(out), self.sm_scale)
            self.step_no += 1
            return out
        plan = self.cache.plan_step(self.req_ids)
        self.cache.apply_cow(plan)
        self.bufs.upload(plan)
        first = self.gs is None
        if first:
            self.gs = GraphStep(self.cache, self.bufs, self.sm_scale, self.R, fused=self.fused_step)
        self.gs.q.copy_(q)
        self.gs.k.copy_(kn)
        self.gs.v.copy_(vn)
        if first or not self.graph:
            self.gs.run_eager()
            if self.graph:
                self.gs.capture()
        else:
            self.gs.replay()
        self.cache.commit_step(self.req_ids)
        self.step_no += 1
        return self.gs.out.clone()

    def error_bits(self) -> int:
        return sum(lc.error_bits() for lc in self.cache.layers)

    # -- oracle ---------------------------------------------------------------
    def history(self, layer: int, i: int, n: int) -> SequenceHistory:
        r = self.req_ids[i]
        h = SequenceHistory(self.Hkv, self.d, self.bs, self.cache.layer_int8[layer])
        pos = torch.arange(n)
        h.append(self.kv(layer, synth.KIND_K, r, pos, "cpu").float().numpy(),
                 self.kv(layer, synth.KIND_V, r, pos, "cpu").float().numpy())
        return h

    def oracle_out(self, layer: int, i: int, step: int, rep: int = 0, hist=None) -> np.ndarray:
        """Oracle output [Hq, d] of sequence i at decode step ``step`` (attention
        call ``layer * R + rep``)."""
        n = self.prior[i] + step + 1
        h = hist if hist is not None else self.history(layer, i, n)
        k, v = h.context()
        q = self.q_for(layer * self.R + rep, step, [self.req_ids[i]], "cpu")[0].float().numpy()
        return decode_attention(q, k, v, self.sm_scale)

    def oracle_steps(self, layer: int, i: int, steps: int, rep: int = 0) -> list:
        """Oracle outputs of sequence i for decode steps 0..steps-1, growing one
        history a token at a time (quantizing at its own fill points)."""
        h = self.history(layer, i, self.prior[i])
        r = self.req_ids[i]
        outs = []
        for t in range(steps):
            p = torch.tensor([self.prior[i] + t])
            h.append(self.kv(layer, synth.KIND_K, r, p, "cpu").float().numpy(),
                     self.kv(layer, synth.KIND_V, r, p, "cpu").float().numpy())
            outs.append(self.oracle_out(layer, i, t, rep, hist=h))
        return outs

    def check_pool_bytes(self, layer: int, i: int, n: int) -> int:
        """Compares the pools of sequence i (first n tokens) with the oracle's
        history byte for byte; returns the number of blocks compared."""
        h = self.history(layer, i, n)
        lc = self.cache.layers[layer]
        int8 = lc.int8
        tab = self.cache.table(self.req_ids[i])
        nf = n // self.bs
        nb = -(-n // self.bs)
        ids = torch.tensor(tab[: (nf if int8 else nb)], dtype=torch.long, device=lc.k_pool.device)
        if int8:
            kp = lc.k_pool[ids].cpu().numpy()
            vp = lc.v_pool[ids].cpu().numpy()
            sc = lc.scales[ids].cpu().numpy()
            for bi in range(nf):
                qk, sk, qv, sv = h.blocks[bi]
                assert np.array_equal(kp[bi], qk), (layer, i, bi, "K codes")
                assert np.array_equal(vp[bi], qv), (layer, i, bi, "V codes")
                assert np.array_equal(sc[bi, :, 0].view(np.uint32), sk.view(np.uint32)), (layer, i, bi, "K scale")
                assert np.array_equal(sc[bi, :, 1].view(np.uint32), sv.view(np.uint32)), (layer, i, bi, "V scale")
            rem = n - nf * self.bs
            if rem:
                slot = self.cache.seqs[self.req_ids[i]].slot
                kr, vr = h.raw()
                kt = lc.k_tail[slot, :, :rem].float().cpu().numpy()
                assert np.array_equal(kt, kr[nf * self.bs:].transpose(1, 0, 2)), (layer, i, "K tail")
                vt = lc.v_tail[slot, :, :rem].float().cpu().numpy()
                assert np.array_equal(vt, vr[nf * self.bs:].transpose(1, 0, 2)), (layer, i, "V tail")
            return nf
        kp = lc.k_pool[ids].float().cpu().numpy()
        vp = lc.v_pool[ids].float().cpu().numpy()
        kr, vr = h.raw()
        for bi in range(nb):
            lo, hi = bi * self.bs, min(n, (bi + 1) * self.bs)
            assert np.array_equal(kp[bi][:, : hi - lo], kr[lo:hi].transpose(1, 0, 2)), (layer, i, bi, "K rows")
            assert np.array_equal(vp[bi][:, : hi - lo], vr[lo:hi].transpose(1, 0, 2)), (layer, i, bi, "V rows")
        return nb
