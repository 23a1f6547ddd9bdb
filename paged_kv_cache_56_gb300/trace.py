"""Continuous-batching trace driver (host control logic around the cache).

Each step ("轻量级推理引擎实战" §2.2, "vLLM核心概念" §3.3): evict the requests
that finished (their private blocks return to the free list, "连续批处理与KV缓存"
§4.2 free), admit waiting requests first-come first-served while free blocks
allow, then run one decode step (append + quantize-on-fill + attention) for
every running request through all layers.

Requests share a system-prompt prefix ("vLLM核心概念" §3.2 / §3.6: a 200-token
system prompt whose blocks every request's table points at): the prefix's
full blocks are written once and attached to every request; its remaining
tokens are copied into each request's own blocks. Token p of a request holds
the prefix's row p when p < prefix_tokens, else the request's own row.

Admission reading: a request needs ceil((prefix + prompt) / bs) - shared
private blocks for its prompt; it is admitted when free blocks cover that plus
one block per running request (the most the next step's appends can take), so
an append never has to wait.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

from . import pkv, synth
from .runtime import PagedKVCache, StepBuffers, prefill, sm_scale_for

PREFIX_SEQ = 10 ** 6  # synthetic sequence id of the shared prefix rows

# Launch configuration of the trace's decode steps: split length in tokens
# (measured best on GB300 among 512..4096 for this workload) and
# programmatic dependent launch between the layers' kernels.
TRACE_SPLIT_TOKENS = 1536
TRACE_PDL = True


@dataclass
class Request:
    rid: int
    arrival: int
    prompt: int
    output: int
    generated: int = 0

    @property
    def length(self) -> int:  # tokens in the cache before the next decode step
        return self.prompt_total + self.generated

    prompt_total: int = 0


class TraceDriver:
    def __init__(self, cache: PagedKVCache, seed: int, num_steps: int, max_running: int = 128,
                 prefix_tokens: int = 200, arrival_rate: float = 2.0, prompt_min: int = 16,
                 prompt_max: int = 4096, mean_output: float = 300.0, split_tokens: int = 0,
                 fused: bool = True):
        self.cache = cache
        self.seed = seed
        self.max_running = max_running
        self.prefix_tokens = prefix_tokens
        self.shared_blocks = prefix_tokens // cache.bs
        self.sm_scale = sm_scale_for(cache.d)
        self.fused = fused
        self.arrivals = [Request(rid, a, p, o) for a, rid, p, o in
                         synth.trace_requests(seed, num_steps, arrival_rate, prompt_min, prompt_max, mean_output)]
        self.waiting: list[Request] = []
        self.running: list[Request] = []
        self.finished: list[Request] = []
        self.step_no = 0
        self._next_arrival = 0
        self.bufs = StepBuffers(cache, max_running, split_tokens, fused_merge=True)
        self.out = torch.empty((cache.L, max_running, cache.hq, cache.d), dtype=torch.bfloat16,
                               device=cache.device)
        self.prefix_ids = []
        self._write_prefix()
        self.descs = pkv.desc_array([lc.desc for lc in cache.layers])

    # -- synthetic rows ------------------------------------------------------
    def rows(self, layer: int, kind: int, rid: int, positions, device=None) -> torch.Tensor:
        """K or V rows of request rid at the given positions (prefix rows below
        prefix_tokens, the request's own rows above)."""
        c = self.cache
        positions = torch.as_tensor(positions, dtype=torch.int64)
        seqs = torch.where(positions < self.prefix_tokens, torch.full_like(positions, PREFIX_SEQ),
                           torch.full_like(positions, rid))
        return synth.kv_rows(self.seed, layer, kind, seqs, positions, c.hkv, c.d, device=device or c.device)

    def q_rows(self, layer: int, rids, step: int, device=None) -> torch.Tensor:
        c = self.cache
        return synth.q_rows(self.seed, layer, step, rids, c.hq, c.d, device=device or c.device)

    def _write_prefix(self) -> None:
        c = self.cache
        if self.shared_blocks == 0:
            return
        c.add_sequence(PREFIX_SEQ, self.shared_blocks)
        self.prefix_ids = c.table(PREFIX_SEQ)
        n = self.shared_blocks * c.bs
        for li in range(c.L):
            pos = torch.arange(n)
            prefill(c, li, [PREFIX_SEQ], [self.rows(li, synth.KIND_K, PREFIX_SEQ, pos)],
                    [self.rows(li, synth.KIND_V, PREFIX_SEQ, pos)])
        c.seqs[PREFIX_SEQ].length = n

    # -- scheduling ----------------------------------------------------------
    def _private_blocks_for(self, total_tokens: int) -> int:
        return -(-total_tokens // self.cache.bs) - self.shared_blocks

    def _admit(self) -> list:
        c = self.cache
        while self._next_arrival < len(self.arrivals) and self.arrivals[self._next_arrival].arrival <= self.step_no:
            self.waiting.append(self.arrivals[self._next_arrival])
            self._next_arrival += 1
        admitted = []
        while self.waiting and len(self.running) < self.max_running and c.free_slots:
            r = self.waiting[0]
            total = self.prefix_tokens + r.prompt
            need = self._private_blocks_for(total)
            if pkv.pkv_num_free(c.alloc) < need + len(self.running) + 1:
                break  # FCFS: the head of the queue waits, nobody overtakes it
            self.waiting.pop(0)
            c.add_sequence(r.rid, need, shared_blocks=self.prefix_ids)
            r.prompt_total = total
            admitted.append(r)
            self.running.append(r)
        if admitted:
            start = self.shared_blocks * c.bs
            for li in range(c.L):
                ks, vs = [], []
                for r in admitted:
                    pos = torch.arange(start, r.prompt_total)
                    ks.append(self.rows(li, synth.KIND_K, r.rid, pos))
                    vs.append(self.rows(li, synth.KIND_V, r.rid, pos))
                prefill(c, li, [r.rid for r in admitted], ks, vs, starts=[start] * len(admitted))
            for r in admitted:
                c.seqs[r.rid].length = r.prompt_total
        return admitted

    def _evict(self) -> list:
        done = [r for r in self.running if r.generated >= r.output]
        for r in done:
            self.cache.remove_sequence(r.rid)
            self.running.remove(r)
            self.finished.append(r)
        return done

    # -- one step ------------------------------------------------------------
    def step(self, events=None):
        """Evict, admit, decode. Returns (running request ids, plan) of the
        decode, or ([], None) when nothing runs. events: optional (start, end)
        CUDA events recorded around the decode kernels."""
        c = self.cache
        self._evict()
        self._admit()
        if not self.running:
            self.step_no += 1
            return [], None
        rids = self.batch_order()
        plan = c.plan_step(rids)
        c.apply_cow(plan)
        self.bufs.upload(plan)
        B = len(rids)
        pos = torch.tensor(plan.positions, dtype=torch.int64)
        b = self.bufs
        inputs = [(self.q_rows(li, rids, self.step_no), self._new_rows(li, synth.KIND_K, rids, pos),
                   self._new_rows(li, synth.KIND_V, rids, pos)) for li in range(c.L)]
        if self.fused:  # the whole step in one native call
            qs = torch.stack([x[0] for x in inputs])
            ks = torch.stack([x[1] for x in inputs])
            vs = torch.stack([x[2] for x in inputs])
            if events is not None:
                events[0].record()
            pkv.pkv_decode_layers(self.descs, qs, ks, vs, b.tab[:B], b.ctx[:B], b.slot[:B], self.sm_scale,
                                  self.out[:, :B], b.split_tokens, b.max_splits, b.ws_o, b.ws_ml, b.ws_count)
            if events is not None:
                events[1].record()
            c.commit_step(rids)
            for r in self.running:
                r.generated += 1
            self.step_no += 1
            return rids, plan
        if events is not None:
            events[0].record()
        for li, lc in enumerate(c.layers):
            q, k, v = inputs[li]
            if self.fused:
                pkv.pkv_decode_step(lc.desc, q, k, v, b.tab[:B], b.ctx[:B], b.slot[:B], self.sm_scale,
                                    self.out[li, :B], b.split_tokens, b.max_splits, b.ws_o, b.ws_ml, b.ws_count)
            else:
                pkv.pkv_append_kv(lc.desc, k, v, b.blk[:B], b.off[:B], b.slot[:B])
                if lc.int8 and (plan.fill_blocks >= 0).any():
                    pkv.pkv_quantize_full_blocks(lc.desc, b.fill[:B], b.slot[:B])
                pkv.pkv_decode_attention(lc.desc, q, b.tab[:B], b.ctx[:B], b.slot[:B], self.sm_scale,
                                         self.out[li, :B], b.split_tokens, b.max_splits, b.ws_o, b.ws_ml,
                                         b.ws_count)
        if events is not None:
            events[1].record()
        c.commit_step(rids)
        for r in self.running:
            r.generated += 1
        self.step_no += 1
        return rids, plan

    def batch_order(self) -> list:
        """Running request ids in the order the step batches them. The decode
        grid starts its CTAs in batch order. The shortest quarter of the
        requests goes first, shortest first: their CTAs do little streaming
        and mostly wait on their start-up loads (context, table, query, tail),
        so they are best started while the previous layer drains and finished
        early, instead of ending the layer. The rest follow longest first, so
        the long sequences start at once and the others fill in behind them."""
        rs = sorted(self.running, key=lambda r: -r.length)
        k = len(rs) // 4
        rs = rs[len(rs) - k:][::-1] + rs[:len(rs) - k]
        return [r.rid for r in rs]

    def _new_rows(self, layer: int, kind: int, rids, positions) -> torch.Tensor:
        c = self.cache
        seqs = torch.tensor(rids, dtype=torch.int64)
        positions = positions.clone()
        seqs = torch.where(positions < self.prefix_tokens, torch.full_like(seqs, PREFIX_SEQ), seqs)
        return synth.kv_rows(self.seed, layer, kind, seqs, positions, c.hkv, c.d, device=c.device)
