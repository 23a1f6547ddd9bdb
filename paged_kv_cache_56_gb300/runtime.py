"""Host-side runtime around the C ABI: per-layer device buffers, the block
allocator, sequence slots, and the per-step control arrays (positions, block
tables, context lengths, fill lists).

Every computation on cache data runs in libpkv.so's kernels; this module only
allocates device memory with torch, keeps host bookkeeping, and calls the
binding. A decode step for B running sequences is:

  1. (host) a sequence at position p with p % block_size == 0 gets a new
     block from the allocator ([D] "连续批处理与KV缓存" §4.2 append_block);
  2. (host -> device) block tables, context lengths, offsets and fill lists;
  3. per layer: append the new K/V rows, quantize the blocks that filled
     (INT8), decode attention (+ split-K merge).
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

from . import pkv


class LayerCache:
    """Device buffers of one layer and the descriptor that points at them."""

    def __init__(self, num_blocks: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                 block_size: int, int8: bool, max_slots: int, device="cuda"):
        self.num_blocks, self.hq, self.hkv, self.d, self.bs = num_blocks, num_q_heads, num_kv_heads, head_dim, block_size
        self.int8 = int8
        shape = (num_blocks, num_kv_heads, block_size, head_dim)
        pool_dtype = torch.int8 if int8 else torch.bfloat16
        self.k_pool = torch.empty(shape, dtype=pool_dtype, device=device)
        self.v_pool = torch.empty(shape, dtype=pool_dtype, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        if int8:
            self.scales = torch.zeros((num_blocks, num_kv_heads, 2), dtype=torch.float32, device=device)
            tail_shape = (max_slots, num_kv_heads, block_size, head_dim)
            self.k_tail = torch.zeros(tail_shape, dtype=torch.bfloat16, device=device)
            self.v_tail = torch.zeros(tail_shape, dtype=torch.bfloat16, device=device)
        else:
            self.scales = self.k_tail = self.v_tail = None
        self.desc = pkv.CacheDesc(
            k_pool=self.k_pool.data_ptr(), v_pool=self.v_pool.data_ptr(),
            scales=self.scales.data_ptr() if int8 else None,
            k_tail=self.k_tail.data_ptr() if int8 else None,
            v_tail=self.v_tail.data_ptr() if int8 else None,
            num_blocks=num_blocks, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
            head_dim=head_dim, block_size=block_size, max_slots=max_slots if int8 else 0,
            dtype=pkv.PKV_DTYPE_INT8 if int8 else pkv.PKV_DTYPE_BF16,
            err_word=self.err.data_ptr())

    def error_bits(self) -> int:
        return int(self.err.item())


def choose_split_tokens(batch: int, num_kv_heads: int, max_ctx: int, block_size: int,
                        num_sms: int, ctas_per_sm: int) -> int:
    """Split length (a multiple of 16 and of block_size) such that the
    (sequence, kv head, split) CTAs of the longest context fit in one wave of
    num_sms * ctas_per_sm resident CTAs; 0 (no split) when one CTA per
    (sequence, kv head) already fills a wave."""
    pairs = batch * num_kv_heads
    slots = num_sms * ctas_per_sm
    splits = slots // max(pairs, 1)
    if splits <= 1 or max_ctx <= 0:
        return 0
    unit = max(16, block_size)
    tok = -(-max_ctx // splits)
    return max(unit, -(-tok // unit) * unit)


def plan_split_tokens(cache: "PagedKVCache", batch: int, max_ctx: int, num_sms: int | None = None) -> int:
    """choose_split_tokens with this cache's measured decode occupancy."""
    if num_sms is None:
        num_sms = torch.cuda.get_device_properties(torch.device(cache.device)).multi_processor_count
    desc = cache.layers[0].desc
    unit = max(16, cache.bs)
    occ = pkv.pkv_decode_ctas_per_sm(desc, unit, cache.max_blocks)
    split = choose_split_tokens(batch, cache.hkv, max_ctx, cache.bs, num_sms, occ)
    if split:
        occ2 = pkv.pkv_decode_ctas_per_sm(desc, split, cache.max_blocks)
        if occ2 < occ:
            split = choose_split_tokens(batch, cache.hkv, max_ctx, cache.bs, num_sms, occ2)
    else:
        occ0 = pkv.pkv_decode_ctas_per_sm(desc, 0, cache.max_blocks)
        if batch * cache.hkv < num_sms * occ0:
            split = choose_split_tokens(batch, cache.hkv, max_ctx, cache.bs, num_sms, occ0)
    return split


@dataclass
class Seq:
    req_id: int
    slot: int
    length: int = 0  # tokens already in the cache


@dataclass
class StepPlan:
    """Host arrays describing one decode step of B sequences."""
    positions: np.ndarray      # [B] token index written this step
    ctx_lens: np.ndarray       # [B] tokens attended over (positions + 1)
    offsets: np.ndarray        # [B] positions % block_size
    block_ids: np.ndarray      # [B] block receiving the new row
    slots: np.ndarray          # [B]
    fill_blocks: np.ndarray    # [B] block that filled this step, or -1
    tables: np.ndarray         # [B, max_blocks]
    tables_changed: bool = True
    cow: list = None           # (old, new) block pairs to copy before the step's writes


class PagedKVCache:
    """L layers of paged cache sharing one allocator and one slot space."""

    def __init__(self, num_layers: int, num_blocks: int, num_q_heads: int, num_kv_heads: int,
                 head_dim: int, block_size: int, int8: bool, max_slots: int, max_blocks_per_seq: int,
                 device="cuda", initial_order=None):
        self.L = num_layers
        self.bs = block_size
        self.hq, self.hkv, self.d = num_q_heads, num_kv_heads, head_dim
        # int8: one flag for every layer, or one per layer -- mixed precision
        # ("轻量级推理引擎实战" §3.2: bf16 for the sensitive first and last
        # layers, INT8 in between); each layer's descriptor carries its dtype
        flags = [bool(int8)] * num_layers if isinstance(int8, (bool, int)) else [bool(x) for x in int8]
        if len(flags) != num_layers:
            raise ValueError("int8 needs one flag per layer")
        self.layer_int8 = flags
        self.int8 = any(flags)  # some layer keeps INT8 blocks: fills are tracked
        self.max_slots = max_slots
        self.max_blocks = max_blocks_per_seq
        self.device = device
        self.layers = [LayerCache(num_blocks, num_q_heads, num_kv_heads, head_dim, block_size, f,
                                  max_slots, device) for f in flags]
        self.alloc = pkv.pkv_allocator_create(num_blocks, block_size, initial_order)
        self.free_slots = list(range(max_slots))
        self.seqs: dict[int, Seq] = {}
        self.forked = False  # set by fork(): only then can a block have several holders

    def close(self):
        if self.alloc is not None:
            pkv.pkv_allocator_destroy(self.alloc)
            self.alloc = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- requests ------------------------------------------------------------
    def add_sequence(self, req_id: int, n_blocks: int = 0, shared_blocks=()) -> Seq:
        if not self.free_slots:
            raise RuntimeError("no free sequence slot")
        pkv.pkv_alloc(self.alloc, req_id, n_blocks)
        if len(shared_blocks):
            pkv.pkv_attach_shared(self.alloc, req_id, list(shared_blocks))
        s = Seq(req_id, self.free_slots.pop(0), 0)
        self.seqs[req_id] = s
        return s

    def fork(self, parent: int, child: int, stream=None) -> Seq:
        """Copy-on-write fork ("vLLM核心概念" §3.2: parallel sampling, beam
        search): the child holds every block of the parent and continues from
        the same length; blocks are copied only when a holder writes into a
        shared one (plan_step). INT8: the partly filled block lives in the
        slot's bf16 tail, which is copied to the child's slot here."""
        if not self.free_slots:
            raise RuntimeError("no free sequence slot")
        p = self.seqs[parent]
        pkv.pkv_fork(self.alloc, parent, child)
        self.forked = True
        s = Seq(child, self.free_slots.pop(0), p.length)
        self.seqs[child] = s
        if self.int8 and p.length % self.bs:
            dev = self.layers[0].k_pool.device
            src = torch.tensor([p.slot], dtype=torch.int32, device=dev)
            dst = torch.tensor([s.slot], dtype=torch.int32, device=dev)
            for lc in self.layers:
                if lc.int8:
                    pkv.pkv_copy_slots(lc.desc, src, dst, stream)
        return s

    def remove_sequence(self, req_id: int) -> None:
        s = self.seqs.pop(req_id)
        pkv.pkv_free(self.alloc, req_id)
        self.free_slots.append(s.slot)

    def table(self, req_id: int) -> list:
        return pkv.pkv_request_table(self.alloc, req_id)

    def stats(self) -> dict:
        """Pool occupancy ("vLLM核心概念" §3.5: blocks used of total): free and
        used blocks, live sequences, and the tokens allocated but not yet
        written (each sequence's tail-block waste, below one block)."""
        free = pkv.pkv_num_free(self.alloc)
        held = set()
        waste = 0
        for r, sq in self.seqs.items():
            t = self.table(r)
            held.update(t)
            waste += len(t) * self.bs - sq.length
        total = self.layers[0].num_blocks
        return dict(blocks_total=total, blocks_free=free, blocks_used=total - free, blocks_referenced=len(held),
                    sequences=len(self.seqs), tail_waste_tokens=waste)

    # -- one decode step -----------------------------------------------------
    def plan_step(self, req_ids, tables_out: np.ndarray | None = None) -> StepPlan:
        """Host part of one decode step: grows block lists where a new block
        starts, and builds the control arrays. Raises PkvError(OOM) if a
        needed block is not available (the caller decides whether to wait)."""
        B = len(req_ids)
        pos = np.empty(B, np.int32)
        blk = np.empty(B, np.int32)
        fill = np.full(B, -1, np.int32)
        slots = np.empty(B, np.int32)
        changed = False
        cow = []
        for i, r in enumerate(req_ids):
            s = self.seqs[r]
            p = s.length
            if p % self.bs == 0 and len(self.table(r)) <= p // self.bs:
                pkv.pkv_append_block(self.alloc, r)
                changed = True
            elif self.forked and p % self.bs:
                # the row goes into a partly filled block: if a fork left it
                # shared, this request takes a private copy first
                pair = pkv.pkv_cow_block(self.alloc, r, p // self.bs)
                if pair is not None:
                    cow.append(pair)
                    changed = True
            pos[i] = p
            slots[i] = s.slot
        tables = pkv.pkv_build_block_tables(self.alloc, req_ids, self.max_blocks, tables_out)
        for i, r in enumerate(req_ids):
            p = int(pos[i])
            blk[i] = tables[i, p // self.bs]
            if self.int8 and (p + 1) % self.bs == 0:
                fill[i] = blk[i]
        return StepPlan(positions=pos, ctx_lens=pos + 1, offsets=pos % self.bs, block_ids=blk,
                        slots=slots, fill_blocks=fill, tables=tables, tables_changed=changed, cow=cow)

    def apply_cow(self, plan: StepPlan, stream=None) -> None:
        """Device half of the plan's copy-on-write: the old blocks' rows into
        the new ones, every layer, before the step writes. An INT8 block that
        has not filled holds no pool data (its rows are in the slot's tail), so
        there is nothing to copy."""
        if not plan.cow or all(self.layer_int8):
            return
        dev = self.layers[0].k_pool.device
        src = torch.tensor([a for a, _ in plan.cow], dtype=torch.int32, device=dev)
        dst = torch.tensor([b for _, b in plan.cow], dtype=torch.int32, device=dev)
        for lc in self.layers:
            if not lc.int8:
                pkv.pkv_copy_blocks(lc.desc, src, dst, stream)

    def commit_step(self, req_ids) -> None:
        for r in req_ids:
            self.seqs[r].length += 1


def sm_scale_for(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)


# ---------------------------------------------------------------------------
# Prefill (untimed setup: writes a prompt's rows with the same two kernels)
# ---------------------------------------------------------------------------

def prefill(cache: PagedKVCache, layer: int, req_ids, k_rows, v_rows, starts=None, stream=None) -> None:
    """Writes rows k_rows[i] / v_rows[i] ([n_i, Hkv, d] bf16, device) of
    sequence req_ids[i] at positions starts[i] .. starts[i]+n_i-1 (starts must
    be multiples of block_size; the sequence must already hold the blocks).
    BF16 cache: one append of all rows. INT8 cache: whole blocks are quantized
    straight from the rows; the trailing partial block goes to the tail."""
    lc = cache.layers[layer]
    bs = cache.bs
    dev = lc.k_pool.device
    starts = [0] * len(req_ids) if starts is None else list(starts)
    tabs = [cache.table(r) for r in req_ids]
    if not lc.int8:
        blk, off = [], []
        for t, s0, k in zip(tabs, starts, k_rows):
            pos = np.arange(s0, s0 + k.shape[0])
            blk.append(np.asarray(t, np.int32)[pos // bs])
            off.append((pos % bs).astype(np.int32))
        if sum(k.shape[0] for k in k_rows) == 0:
            return
        pkv.pkv_append_kv(lc.desc, torch.cat(list(k_rows)).contiguous(), torch.cat(list(v_rows)).contiguous(),
                          torch.from_numpy(np.concatenate(blk)).to(dev), torch.from_numpy(np.concatenate(off)).to(dev),
                          None, stream)
        return
    fk, fv, fb, tk, tv, ts, to = [], [], [], [], [], [], []
    for r, t, s0, k, v in zip(req_ids, tabs, starts, k_rows, v_rows):
        if s0 % bs:
            raise ValueError("prefill start must be a multiple of block_size")
        n = k.shape[0]
        nf = n // bs
        if nf:
            fk.append(k[: nf * bs])
            fv.append(v[: nf * bs])
            fb.extend(t[s0 // bs: s0 // bs + nf])
        if n % bs:
            tk.append(k[nf * bs:])
            tv.append(v[nf * bs:])
            ts.extend([cache.seqs[r].slot] * (n % bs))
            to.extend(range(n % bs))
    if fb:
        pkv.pkv_quantize_blocks_from(lc.desc, torch.cat(fk).contiguous(), torch.cat(fv).contiguous(),
                                     torch.tensor(fb, dtype=torch.int32, device=dev), stream)
    if ts:
        pkv.pkv_append_kv(lc.desc, torch.cat(tk).contiguous(), torch.cat(tv).contiguous(), None,
                          torch.tensor(to, dtype=torch.int32, device=dev),
                          torch.tensor(ts, dtype=torch.int32, device=dev), stream)


# ---------------------------------------------------------------------------
# Decode steps
# ---------------------------------------------------------------------------

class StepBuffers:
    """Device-side control arrays (and split-K workspace) of decode steps for
    up to max_batch sequences; pinned host mirrors make the uploads async."""

    def __init__(self, cache: PagedKVCache, max_batch: int, split_tokens: int = 0, fused_merge: bool = True):
        dev = cache.device
        self.cache = cache
        self.max_batch = max_batch
        self.split_tokens = split_tokens
        mb = cache.max_blocks
        self.max_splits = -(-(mb * cache.bs) // split_tokens) if split_tokens else 0
        def pair(shape):
            return (torch.zeros(shape, dtype=torch.int32).pin_memory(),
                    torch.zeros(shape, dtype=torch.int32, device=dev))
        self.h_ctx, self.ctx = pair(max_batch)
        self.h_off, self.off = pair(max_batch)
        self.h_blk, self.blk = pair(max_batch)
        self.h_slot, self.slot = pair(max_batch)
        self.h_fill, self.fill = pair(max_batch)
        self.h_tab, self.tab = pair((max_batch, mb))
        if split_tokens:
            self.ws_o = torch.empty(max_batch * cache.hq * self.max_splits * cache.d, dtype=torch.float32, device=dev)
            self.ws_ml = torch.empty(max_batch * cache.hq * self.max_splits * 2, dtype=torch.float32, device=dev)
            # arrival counters of the fused split-K merge (kept at zero between calls)
            self.ws_count = (torch.zeros(max_batch * cache.hkv, dtype=torch.int32, device=dev)
                             if fused_merge else None)
        else:
            self.ws_o = self.ws_ml = self.ws_count = None
        self.B = 0
        self.copied = torch.cuda.Event()  # the last upload's copies have run
        self.copied.record()

    def upload(self, plan: StepPlan) -> None:
        B = len(plan.positions)
        if B > self.max_batch:
            raise ValueError("batch larger than the step buffers")
        self.B = B
        self.copied.synchronize()  # do not overwrite pinned data a pending copy still reads
        self.h_ctx[:B].numpy()[:] = plan.ctx_lens
        self.h_off[:B].numpy()[:] = plan.offsets
        self.h_blk[:B].numpy()[:] = plan.block_ids
        self.h_slot[:B].numpy()[:] = plan.slots
        self.h_fill[:B].numpy()[:] = plan.fill_blocks
        for h, d in ((self.h_ctx, self.ctx), (self.h_off, self.off), (self.h_blk, self.blk),
                     (self.h_slot, self.slot), (self.h_fill, self.fill)):
            d[:B].copy_(h[:B], non_blocking=True)
        self.h_tab[:B].numpy()[:] = plan.tables
        self.tab[:B].copy_(self.h_tab[:B], non_blocking=True)
        self.copied.record()


def run_layers(cache: PagedKVCache, bufs: StepBuffers, q, k_new, v_new, out, sm_scale: float,
               quantize: str = "auto", plan: StepPlan | None = None, stream=None) -> None:
    """Kernel launches of one decode step for bufs.B sequences: per layer l,
    append k_new[l], v_new[l] ([B, Hkv, d]), quantize filled blocks (INT8),
    attend with q[l] ([B, Hq, d]) into out[l] ([B, Hq, d]).

    quantize="auto" launches the quantize kernel only when the plan has a
    filled block; "always" launches it every step over a -1-padded list (the
    form a captured CUDA graph needs)."""
    B = bufs.B
    for li, lc in enumerate(cache.layers):
        pkv.pkv_append_kv(lc.desc, k_new[li], v_new[li], bufs.blk[:B], bufs.off[:B], bufs.slot[:B], stream)
        if lc.int8 and (quantize == "always" or (plan is not None and (plan.fill_blocks >= 0).any())):
            pkv.pkv_quantize_full_blocks(lc.desc, bufs.fill[:B], bufs.slot[:B], stream)
        pkv.pkv_decode_attention(lc.desc, q[li], bufs.tab[:B], bufs.ctx[:B], bufs.slot[:B], sm_scale, out[li],
                                 bufs.split_tokens, bufs.max_splits, bufs.ws_o, bufs.ws_ml, bufs.ws_count, stream)


def decode_step(cache: PagedKVCache, bufs: StepBuffers, req_ids, q, k_new, v_new, out, sm_scale: float,
                stream=None) -> StepPlan:
    """Host plan + upload + kernels of one decode step; advances the sequences."""
    plan = cache.plan_step(req_ids)
    cache.apply_cow(plan, stream)
    bufs.upload(plan)
    run_layers(cache, bufs, q, k_new, v_new, out, sm_scale, "auto", plan, stream)
    cache.commit_step(req_ids)
    return plan


class GraphStep:
    """The kernel launches of one decode step, captured once as a CUDA graph
    ("离开 N 卡后的真实世界" §2: graph capture turns a decode step's dozens of
    small launches into one submission).

    The graph reads its inputs from static device buffers -- ``q`` [L*R, B,
    Hq, d], ``k``/``v`` [L, B, Hkv, d] -- and the StepBuffers control arrays,
    and writes ``out`` [L*R, B, Hq, d]; each layer's attention runs R times
    (R > 1 re-reads the same layer's cache with R different queries). The
    quantize kernel is always launched over a -1-padded fill list so that the
    graph does not change from step to step. The batch size is fixed at
    capture time.
    """

    def __init__(self, cache: PagedKVCache, bufs: StepBuffers, sm_scale: float, repeat: int = 1,
                 fused: bool = True):
        self.cache, self.bufs, self.sm_scale, self.R = cache, bufs, sm_scale, repeat
        self.fused = fused  # one pkv_decode_step per layer instead of append + quantize + attention
        B, dev = bufs.B, cache.device
        if B == 0:
            raise ValueError("upload a plan before capturing")
        L = cache.L
        self.q = torch.zeros((L * repeat, B, cache.hq, cache.d), dtype=torch.bfloat16, device=dev)
        self.k = torch.zeros((L, B, cache.hkv, cache.d), dtype=torch.bfloat16, device=dev)
        self.v = torch.zeros((L, B, cache.hkv, cache.d), dtype=torch.bfloat16, device=dev)
        self.out = torch.zeros((L * repeat, B, cache.hq, cache.d), dtype=torch.bfloat16, device=dev)
        self.graph = None
        self.attn_graph = None

    def launches_per_step(self) -> int:
        per_attn = 2 if (self.bufs.split_tokens and self.bufs.ws_count is None) else 1
        if self.fused:
            return self.cache.L * self.R * per_attn
        return sum(1 + int(f) + self.R * per_attn for f in self.cache.layer_int8)

    def _layers(self, attention_only: bool = False) -> None:
        c, b = self.cache, self.bufs
        B = b.B
        for li, lc in enumerate(c.layers):
            fused_here = self.fused and not attention_only
            if not attention_only and not self.fused:
                pkv.pkv_append_kv(lc.desc, self.k[li], self.v[li], b.blk[:B], b.off[:B], b.slot[:B])
                if lc.int8:
                    pkv.pkv_quantize_full_blocks(lc.desc, b.fill[:B], b.slot[:B])
            for r in range(self.R):
                qi = li * self.R + r
                if fused_here and r == 0:
                    pkv.pkv_decode_step(lc.desc, self.q[qi], self.k[li], self.v[li], b.tab[:B], b.ctx[:B],
                                        b.slot[:B], self.sm_scale, self.out[qi], b.split_tokens, b.max_splits,
                                        b.ws_o, b.ws_ml, b.ws_count)
                else:
                    pkv.pkv_decode_attention(lc.desc, self.q[qi], b.tab[:B], b.ctx[:B], b.slot[:B],
                                             self.sm_scale, self.out[qi], b.split_tokens, b.max_splits, b.ws_o,
                                             b.ws_ml, b.ws_count)

    def run_eager(self) -> None:
        self._layers()

    def capture(self) -> None:
        """Captures the step (and an attention-only variant used for timing).
        Call after one eager step so every kernel attribute is already set."""
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._layers()
        self.attn_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.attn_graph):
            self._layers(attention_only=True)
        torch.cuda.synchronize()

    def replay(self) -> None:
        self.graph.replay()


class PipelinedSteps:
    """Decode steps fed from host memory with the transfers hidden behind
    compute: two sets of step buffers, each with its own captured step graph,
    take turns. Step s uploads its control arrays and its q / k / v on one
    copy stream while step s-1 computes, and returns its outputs to the host
    on a second copy stream (so that the next upload never queues behind a
    return) while step s+1 computes. The steps themselves run in
    order on the caller's stream, so the results are those of GraphStep step
    by step. The first use of each set runs eagerly and captures its graph."""

    def __init__(self, cache: PagedKVCache, max_batch: int, split_tokens: int, sm_scale: float, repeat: int = 1,
                 fused_merge: bool = True):
        self.cache, self.sm_scale, self.R = cache, sm_scale, repeat
        self.sets = [StepBuffers(cache, max_batch, split_tokens, fused_merge) for _ in range(2)]
        self.graphs = [None, None]
        self.copy = torch.cuda.Stream(device=cache.device)      # host -> device
        self.back = torch.cuda.Stream(device=cache.device)      # device -> host
        self.ready = [torch.cuda.Event(), torch.cuda.Event()]     # a set's inputs are on the device
        self.done = [torch.cuda.Event(), torch.cuda.Event()]      # a set's step has run
        self.returned = [torch.cuda.Event(), torch.cuda.Event()]  # a set's outputs are on the host
        for e in self.done + self.returned:
            e.record()
        self.n = 0

    def step(self, req_ids, q, k, v, out=None) -> StepPlan:
        """One decode step. q [L*R, B, Hq, d], k / v [L, B, Hkv, d]: pinned host
        (or device) bf16; out: pinned host bf16 [L*R, B, Hq, d] that receives
        the step's outputs, or None to leave them in ``last_out()``. Host
        buffers must stay untouched until ``finish()`` (or until the same set
        comes round again, two steps later)."""
        i = self.n & 1
        bufs = self.sets[i]
        compute = torch.cuda.current_stream()
        plan = self.cache.plan_step(req_ids)
        self.cache.apply_cow(plan, compute)
        with torch.cuda.stream(self.copy):
            self.copy.wait_event(self.done[i])      # the set's previous step has read its buffers
            self.copy.wait_event(self.returned[i])  # ... and its outputs have left
            bufs.upload(plan)
            gs = self.graphs[i]
            if gs is None:
                gs = GraphStep(self.cache, bufs, self.sm_scale, self.R)
            gs.q.copy_(q, non_blocking=True)
            gs.k.copy_(k, non_blocking=True)
            gs.v.copy_(v, non_blocking=True)
            self.ready[i].record(self.copy)
        compute.wait_event(self.ready[i])
        if self.graphs[i] is None:
            gs.run_eager()
            self.graphs[i] = gs
            self.done[i].record(compute)
            gs.capture()  # synchronises: the eager step is complete
        else:
            gs.replay()
            self.done[i].record(compute)
        if out is not None:
            with torch.cuda.stream(self.back):
                self.back.wait_event(self.done[i])
                out.copy_(gs.out, non_blocking=True)
                self.returned[i].record(self.back)
        self.cache.commit_step(req_ids)
        self.last = i
        self.n += 1
        return plan

    def last_out(self) -> torch.Tensor:
        """Device outputs of the latest step (valid on the caller's stream)."""
        return self.graphs[self.last].out

    def finish(self) -> None:
        """Makes the caller's stream wait for every transfer issued so far."""
        for st in (self.copy, self.back):
            ev = torch.cuda.Event()
            ev.record(st)
            torch.cuda.current_stream().wait_event(ev)
