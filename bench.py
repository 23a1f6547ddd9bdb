#!/usr/bin/env python
"""Decode-step benchmark of the paged KV cache on GB300.

A step is one decode step of every running sequence through all layers:
host block allocation and tables, their upload, then per layer append +
quantize-on-fill + decode attention (+ split-K merge). Inputs are seeded
synthetic rows, generated on the device before timing; the KV working set of
a step (1.84 GB for the default workload) is far larger than L2, so no flush
is needed between steps.

Default workload: GQA TTS-talker decode -- 28 layers, 4 sequences x 8000
context tokens, Hq=16, Hkv=8, d=128, 16-token blocks, INT8 cache with a bf16
tail, per-head scales U(0.1, 4). Other workloads: --workload mha7b | long_bf16
| long_int8 | tiny.

Metric: KV GB/s = algorithmic bytes the attention must read per step / step
time, plus decode tokens/s. ``--impl reference`` times the CPU oracle on a
bounded sample of the same workload instead.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOADS = {
    # name: layers, batch, prior tokens, Hq, Hkv, d, block, pool blocks/layer, int8, head scale, outliers, repeat
    "tts_talker": dict(L=28, B=4, prior=8000, Hq=16, Hkv=8, d=128, bs=16, num_blocks=2048, int8=True,
                       head_scale=True, outliers=False, repeat=1,
                       desc="GQA TTS-talker decode: 28 layers, 4 x 8000 ctx, Hq=16 Hkv=8 d=128, bs=16, INT8"),
    "mha7b": dict(L=32, B=100, prior=1024, Hq=32, Hkv=32, d=128, bs=16, num_blocks=8192, int8=False,
                  head_scale=False, outliers=False, repeat=1,
                  desc="MHA 7B-class decode: 32 layers, 100 x 1024 ctx, 32 heads d=128, bs=16, bf16"),
    "long_bf16": dict(L=1, B=8, prior=32768, Hq=32, Hkv=8, d=128, bs=64, num_blocks=4200, int8=False,
                      head_scale=False, outliers=True, repeat=32,
                      desc="long-context split-K: 8 x 32768 ctx, Hq=32 Hkv=8 d=128, bs=64, bf16, 1 layer x32"),
    "long_int8": dict(L=1, B=8, prior=32768, Hq=32, Hkv=8, d=128, bs=64, num_blocks=4200, int8=True,
                      head_scale=False, outliers=True, repeat=32,
                      desc="long-context split-K: 8 x 32768 ctx, Hq=32 Hkv=8 d=128, bs=64, INT8, 1 layer x32"),
    "trace": dict(L=32, B=128, prior=0, Hq=32, Hkv=8, d=128, bs=16, num_blocks=8192, int8=True,
                  head_scale=False, outliers=False, repeat=1, steps=200,
                  desc="continuous-batching trace: 200 steps, <=128 running, Poisson(2) arrivals, prompts "
                       "log-uniform [16,4096], outputs geometric mean 300, 200-token shared prefix, Hq=32 Hkv=8 "
                       "d=128, bs=16, INT8, 32 layers"),
    "tiny": dict(L=1, B=4, prior=[1, 17, 33, 100], Hq=4, Hkv=2, d=64, bs=16, num_blocks=64, int8=True,
                 head_scale=False, outliers=False, repeat=1,
                 desc="tiny correctness case: 1 layer, ctx {1,17,33,100}, Hq=4 Hkv=2 d=64, bs=16"),
}
SEED = 1234


def _code_only(text: str) -> str:
    """C/C++/CUDA source without comments and with whitespace runs collapsed:
    what the compiler sees, so that editing a comment keeps the hash."""
    import re
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":  # string or character literal, copied as is
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return re.sub(r"\s+", " ", "".join(out)).strip()


def kernel_source_hash() -> str:
    """sha256 over the code (comments and whitespace aside) of the CUDA/C++
    sources and the C header: what an ncu capture measured."""
    import glob
    import hashlib
    h = hashlib.sha256()
    files = sorted(glob.glob(os.path.join(ROOT, "paged_kv_cache_56_gb300", "csrc", "*")) +
                   glob.glob(os.path.join(ROOT, "include", "*.h")))
    for f in files:
        with open(f, encoding="utf-8") as fh:
            h.update(os.path.basename(f).encode() + b"\0" + _code_only(fh.read()).encode())
    return h.hexdigest()


def measured_traffic(workload: str):
    """DRAM bytes (read + write) per launch of the decode kernel from the ncu
    capture recorded in profiles/dram_traffic.json, or None when the kernel
    sources have changed since that capture."""
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("source_sha256") != kernel_source_hash():
        return None
    ent = rec.get("workloads", {}).get(workload)
    return None if ent is None else int(ent["dram_bytes_per_launch"])


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# byte accounting (algorithmic: what the method must read/write, nothing else)
# ---------------------------------------------------------------------------

def attention_bytes(ctx_lens, Hq, Hkv, d, bs, int8) -> int:
    """Bytes one attention call must move: the KV of every attended token
    (int8 full blocks at 1 B/elem plus one fp32 scale per block, head and
    K|V; bf16 tail or bf16 cache at 2 B/elem), one int32 table entry per
    block, q in and out (bf16)."""
    total = 0
    for n in ctx_lens:
        n = int(n)
        nblk = -(-n // bs)
        if int8:
            full = (n // bs) * bs
            total += full * Hkv * 2 * d * 1 + (n - full) * Hkv * 2 * d * 2 + (n // bs) * Hkv * 2 * 4
        else:
            total += n * Hkv * 2 * d * 2
        total += nblk * 4 + Hq * d * 2 * 2
    return total


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.5)
        except Exception:
            self.proc = None

    def stop(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        if self.proc is None:
            return out
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return out
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for nm, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        out["sm_mhz"] = statistics.median(float(r[1]) for r in rows)
        out["sm_max_mhz"] = max(float(r[2]) for r in rows)
        out["reasons"] = sorted(reasons)
        out["samples"] = len(rows)
        return out


# ---------------------------------------------------------------------------
# the device arm
# ---------------------------------------------------------------------------

class Bench:
    def __init__(self, wl: dict, device: str, steps_total: int, split=None, fused_merge=True):
        from paged_kv_cache_56_gb300 import synth
        from paged_kv_cache_56_gb300.runtime import PagedKVCache, StepBuffers, plan_split_tokens, prefill

        self.wl = wl
        self.synth = synth
        self.device = device
        L, B, Hq, Hkv, d, bs = wl["L"], wl["B"], wl["Hq"], wl["Hkv"], wl["d"], wl["bs"]
        prior = wl["prior"] if isinstance(wl["prior"], list) else [wl["prior"]] * B
        self.prior = prior
        self.reqs = list(range(1000, 1000 + B))
        self.sm_scale = 1.0 / math.sqrt(d)
        max_blocks = -(-(max(prior) + steps_total + 1) // bs)
        need = sum(-(-(n + steps_total + 1) // bs) for n in prior)
        if need > wl["num_blocks"]:
            raise SystemExit(f"{steps_total} decode steps need {need} blocks per layer; the workload's pool "
                             f"holds {wl['num_blocks']} (reduce --steps / --warmup / --e2e-steps)")
        self.cache = PagedKVCache(L, wl["num_blocks"], Hq, Hkv, d, bs, wl["int8"], max_slots=B,
                                  max_blocks_per_seq=max_blocks, device=device,
                                  initial_order=synth.permutation(SEED, wl["num_blocks"]))
        self.split = plan_split_tokens(self.cache, B, max(prior) + steps_total + 1) if split is None else split
        self.bufs = StepBuffers(self.cache, B, self.split, fused_merge=fused_merge)
        for r, n in zip(self.reqs, prior):
            self.cache.add_sequence(r, -(-n // bs))
        for li in range(L):
            ks = [self.kv(li, synth.KIND_K, r, torch.arange(n, device=device)) for r, n in zip(self.reqs, prior)]
            vs = [self.kv(li, synth.KIND_V, r, torch.arange(n, device=device)) for r, n in zip(self.reqs, prior)]
            prefill(self.cache, li, self.reqs, ks, vs)
            del ks, vs
        for r, n in zip(self.reqs, prior):
            self.cache.seqs[r].length = n
        torch.cuda.synchronize()
        self.R = wl["repeat"]
        self.launches = 0

    def kv_mult(self, layer, kind):
        wl, s = self.wl, self.synth
        if wl["outliers"]:
            return s.outlier_multipliers(SEED, layer, kind, wl["Hkv"], wl["d"])
        if wl["head_scale"]:
            return s.head_multipliers(SEED, layer, kind, wl["Hkv"])
        return None

    def kv(self, layer, kind, req, pos):
        wl = self.wl
        return self.synth.kv_rows(SEED, layer, kind, req, pos, wl["Hkv"], wl["d"], mult=self.kv_mult(layer, kind),
                                  device=self.device)

    def step_inputs(self, step: int):
        """Device tensors q [L*R, B, Hq, d], k/v [L, B, Hkv, d] for decode step ``step``."""
        wl, s = self.wl, self.synth
        pos = torch.tensor([n + step for n in self.prior], dtype=torch.int64, device=self.device)
        qm = lambda li: s.head_multipliers(SEED, li, s.KIND_Q, wl["Hq"]) if wl["head_scale"] else None
        q = torch.stack([s.q_rows(SEED, li, step, self.reqs, wl["Hq"], wl["d"], mult=qm(li), device=self.device)
                         for li in range(wl["L"] * self.R)])
        k = torch.stack([self.kv(li, s.KIND_K, self.reqs, pos) for li in range(wl["L"])])
        v = torch.stack([self.kv(li, s.KIND_V, self.reqs, pos) for li in range(wl["L"])])
        return q, k, v

    def step(self, gs, q, k, v, graph: bool):
        """One decode step: host plan + control uploads, this step's inputs
        into the graph's static buffers, then the layer loop."""
        plan = self.cache.plan_step(self.reqs)
        self.bufs.upload(plan)
        gs.q.copy_(q, non_blocking=True)
        gs.k.copy_(k, non_blocking=True)
        gs.v.copy_(v, non_blocking=True)
        if graph:
            gs.replay()
        else:
            gs.run_eager()
        self.cache.commit_step(self.reqs)
        return plan


def run_trace(args, wl):
    """The continuous-batching trace: the first `warmup` steps fill the
    system, the next `steps` are timed. Only the decode kernels of each step
    are inside the CUDA events (admission prefill is setup, not the path)."""
    from paged_kv_cache_56_gb300 import pkv, synth
    from paged_kv_cache_56_gb300.runtime import PagedKVCache
    from paged_kv_cache_56_gb300.trace import TRACE_PDL, TRACE_SPLIT_TOKENS, TraceDriver

    pkv.pkv_set_programmatic_launch(TRACE_PDL and not args.no_pdl)
    total_steps = args.warmup + args.steps
    bs = wl["bs"]
    cache = PagedKVCache(wl["L"], wl["num_blocks"], wl["Hq"], wl["Hkv"], wl["d"], bs, wl["int8"],
                         max_slots=wl["B"] + 1, max_blocks_per_seq=-(-(200 + 4096 + total_steps + 16) // bs),
                         device=f"cuda:{torch.cuda.current_device()}",
                         initial_order=synth.permutation(SEED, wl["num_blocks"]))
    split = args.split if args.split is not None else TRACE_SPLIT_TOKENS
    drv = TraceDriver(cache, SEED, total_steps, max_running=wl["B"], split_tokens=split)
    for _ in range(args.warmup):
        drv.step()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    evs, nbytes, ntok, launches = [], 0, 0, 0
    for _ in range(args.steps):
        ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        rids, plan = drv.step(events=ev)
        if rids:
            evs.append(ev)
            nbytes += attention_bytes(plan.ctx_lens, wl["Hq"], wl["Hkv"], wl["d"], bs, wl["int8"]) * wl["L"]
            ntok += len(rids)
            launches += wl["L"]
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = sum(a.elapsed_time(b) for a, b in evs)
    if sum(lc.error_bits() for lc in cache.layers):
        raise RuntimeError("device error bits set")
    return dict(ms=ms, nbytes=nbytes, ntok=ntok, launches=launches, clocks=clk, split=split,
                running=len(drv.running), finished=len(drv.finished), pool=cache.stats())


def max_over_ranks(ms: float, world: int) -> float:
    """The job's time: the slowest rank's timed region (every rank runs the
    same number of steps on its own replica)."""
    if world <= 1:
        return ms
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: the bytes all ranks processed over the job's time."""
    return bytes_per_rank * world / (ms * 1e-3) / 1e9


def run_device(args, wl, rank, world):
    from paged_kv_cache_56_gb300.runtime import GraphStep, PipelinedSteps

    device = f"cuda:{torch.cuda.current_device()}"
    steps_total = args.warmup + args.steps + args.e2e_steps
    bench = Bench(wl, device, steps_total, split=args.split, fused_merge=not args.separate_merge)
    L, R, B = wl["L"], wl["repeat"], wl["B"]
    Hq, Hkv, d, bs = wl["Hq"], wl["Hkv"], wl["d"], wl["bs"]
    graph = not args.eager
    from paged_kv_cache_56_gb300 import pkv
    pkv.pkv_set_programmatic_launch(not args.no_pdl)
    # inputs for every step, resident in HBM before timing
    inputs = [bench.step_inputs(s) for s in range(args.warmup + args.steps)]
    # Graphs: the runtime's PipelinedSteps (control uploads and input copies on
    # a copy stream, two alternating captured step graphs; the first warm-up
    # steps capture them). Eager: one GraphStep run kernel by kernel.
    pipe = gs = None
    if graph:
        pipe = PipelinedSteps(bench.cache, B, bench.split, bench.sm_scale, R, fused_merge=not args.separate_merge)
    run = (lambda s, q, k, v, out=None: pipe.step(bench.reqs, q, k, v, out)) if graph else None
    for s in range(args.warmup):
        if graph:
            run(s, *inputs[s])
            continue
        if gs is None:
            plan = bench.cache.plan_step(bench.reqs)
            bench.bufs.upload(plan)
            gs = GraphStep(bench.cache, bench.bufs, bench.sm_scale, R)
            q, k, v = inputs[s]
            gs.q.copy_(q)
            gs.k.copy_(k)
            gs.v.copy_(v)
            gs.run_eager()
            bench.cache.commit_step(bench.reqs)
        else:
            bench.step(gs, *inputs[s], False)
    if graph:
        pipe.finish()
    torch.cuda.synchronize()

    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    ctx_hist = []
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    start.record()
    for s in range(args.steps):
        x = inputs[args.warmup + s]
        plan = run(s, *x) if graph else bench.step(gs, *x, False)
        ctx_hist.append(plan.ctx_lens.copy())
    if graph:
        pipe.finish()
    stop.record()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    last = pipe.graphs[pipe.last] if graph else gs
    launches = last.launches_per_step() * args.steps
    ms = start.elapsed_time(stop)

    # roofline: the step's kernels alone (one pkv_decode_step per layer and
    # repeat), replayed back to back on the launching stream and timed with
    # CUDA events. Re-running the last step's launches with its unchanged
    # control arrays is idempotent: the same row is rewritten and a block that
    # filled is quantized again to the same bytes.
    attn_reps = max(3, min(200, int(200.0 / max(ms / args.steps, 1e-3))))
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record()
    for _ in range(attn_reps):
        if graph:
            last.graph.replay()
        else:
            last._layers()
    a1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    attn_call_ms = a0.elapsed_time(a1) / (attn_reps * L * R)
    attn_bytes = attention_bytes(ctx_hist[-1], Hq, Hkv, d, bs, wl["int8"])
    ms = max_over_ranks(ms, world)
    step_bytes = sum(attention_bytes(c, Hq, Hkv, d, bs, wl["int8"]) for c in ctx_hist) * L * R
    err = sum(lc.error_bits() for lc in bench.cache.layers)
    if err:
        raise RuntimeError(f"device error bits {err}")

    # e2e: the same steps through host (pinned) buffers: every step's q/k/v go
    # host -> device and its outputs device -> host inside the timed region
    # (with graphs, overlapped with the neighbouring steps' compute by
    # PipelinedSteps; eagerly, each step copies in, runs and copies out).
    e2e = None
    if args.e2e_steps > 0:
        base = args.warmup + args.steps
        host_in = []
        for s in range(args.e2e_steps):
            q, k, v = bench.step_inputs(base + s)
            host_in.append(tuple(t.cpu().pin_memory() for t in (q, k, v)))
        houts = [torch.empty(last.out.shape, dtype=last.out.dtype).pin_memory() for _ in range(2)]
        e_ctx = []
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for s in range(args.e2e_steps):
            if graph:
                plan = run(s, *host_in[s], houts[s % 2])
            else:
                plan = bench.step(gs, *host_in[s], False)
                houts[0].copy_(gs.out, non_blocking=True)
            e_ctx.append(plan.ctx_lens.copy())
        if graph:
            pipe.finish()
        t1.record()
        torch.cuda.synchronize()
        e_ms = max_over_ranks(t0.elapsed_time(t1), world)
        e_bytes = sum(attention_bytes(c, Hq, Hkv, d, bs, wl["int8"]) for c in e_ctx) * L * R
        h2d = sum(t.numel() * t.element_size() for t in host_in[0])
        e2e = {"value": round(job_gbs(e_bytes, world, e_ms), 2), "unit": "GB/s",
               "tokens_per_s": round(B * world * args.e2e_steps / (e_ms * 1e-3), 1),
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(houts[0].numel() * houts[0].element_size()),
               "ms_per_step": round(e_ms / args.e2e_steps, 4)}
    return dict(ms=ms, attn_call_ms=attn_call_ms, attn_bytes=attn_bytes, step_bytes=step_bytes, clocks=clk,
                launches=launches, split=bench.split, ctx=(int(ctx_hist[0].min()), int(ctx_hist[-1].max())),
                e2e=e2e, graph=graph)


# ---------------------------------------------------------------------------
# the oracle arm (CPU)
# ---------------------------------------------------------------------------

def _oracle_contexts(wl) -> list:
    """Context lengths the CPU sample decodes from: the workload's own, or for
    the trace, the shared prefix plus the first requests' prompts."""
    if wl.get("steps"):  # the trace: 200-token prefix + log-uniform prompts
        from paged_kv_cache_56_gb300 import synth
        return [200 + p for _, _, p, _ in synth.trace_requests(SEED, 40)[:16]]
    return wl["prior"] if isinstance(wl["prior"], list) else [wl["prior"]] * wl["B"]


_POOL_BARRIER = None


def _pool_init(barrier):
    global _POOL_BARRIER
    _POOL_BARRIER = barrier


def _f32(a: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp32 values (exact)."""
    return (a.astype(np.uint32) << 16).view(np.float32)


def _oracle_task(task):
    """One worker's share of the CPU sample. For each (sequence, kv head) unit
    a one-head history of the context is built (untimed); then, after a
    barrier with the other workers (sync), each step appends the unit's new
    row and runs the oracle's context read and fp64 attention for the kv
    head's query group. Returns (seconds in the timed region, steps done,
    bytes, unit-steps)."""
    meta, units, steps, budget_s, sync = task
    from oracle.attention import decode_attention
    from oracle.cache import SequenceHistory
    d, bs, int8, G = meta["d"], meta["bs"], meta["int8"], meta["G"]
    work = []
    for n, k, v, qs in units:
        hist = SequenceHistory(1, d, bs, int8)
        hist.append(_f32(k[:n]), _f32(v[:n]))
        work.append((n, hist, _f32(k[n:]), _f32(v[n:]), _f32(qs)))
    sm = 1.0 / math.sqrt(d)
    if sync:
        _POOL_BARRIER.wait()
    done_bytes = done = 0
    t0 = time.perf_counter()
    s = 0
    while s < steps:
        for n, hist, kn, vn, qs in work:
            hist.append(kn[s:s + 1], vn[s:s + 1])
            kc, vc = hist.context()
            decode_attention(qs[s], kc, vc, sm)
            done_bytes += attention_bytes([n + s + 1], G, 1, d, bs, int8)
            done += 1
        s += 1
        if budget_s is not None and time.perf_counter() - t0 > budget_s:
            break
    return time.perf_counter() - t0, s, done_bytes, done


def oracle_baseline(wl, budget_s: float = 10.0, max_units: int = 64, max_steps: int = 64):
    """Times the oracle on the GPU machine's host cores over a bounded sample of
    the workload: layer 0 of the first sequences, every kv head of each, as
    (sequence, kv head) work units (inputs generated here, untimed). First one
    single-threaded worker runs all units step after step until ~budget_s
    have passed (at most max_steps steps); then one single-threaded worker
    per host core runs the same steps of the units dealt out among them
    (spawned processes; numpy / BLAS held to one thread each). Returns both
    throughputs (KV GB/s over the units' algorithmic bytes; decode tokens/s of
    whole steps, i.e. layer 0's rate divided by the layers a step runs), the
    worker count and the sample."""
    import multiprocessing as mp
    from paged_kv_cache_56_gb300 import synth
    Hq, Hkv, d = wl["Hq"], wl["Hkv"], wl["d"]
    G = Hq // Hkv
    ctxs = _oracle_contexts(wl)
    nseq = min(len(ctxs), max(1, max_units // Hkv))
    mult = lambda kind: (synth.outlier_multipliers(SEED, 0, kind, Hkv, d) if wl["outliers"] else
                         synth.head_multipliers(SEED, 0, kind, Hkv) if wl["head_scale"] else None)
    qm = synth.head_multipliers(SEED, 0, synth.KIND_Q, Hq) if wl["head_scale"] else None
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    units = []
    for b in range(nseq):
        n, rid = ctxs[b], 1000 + b
        pos = torch.arange(n + max_steps)
        k = bits(synth.kv_rows(SEED, 0, synth.KIND_K, rid, pos, Hkv, d, mult=mult(synth.KIND_K)))
        v = bits(synth.kv_rows(SEED, 0, synth.KIND_V, rid, pos, Hkv, d, mult=mult(synth.KIND_V)))
        q = bits(synth.q_rows(SEED, 0, torch.arange(max_steps), [rid] * max_steps, Hq, d, mult=qm))
        for h in range(Hkv):
            units.append((n, np.ascontiguousarray(k[:, h]), np.ascontiguousarray(v[:, h]),
                          np.ascontiguousarray(q[:, h * G:(h + 1) * G])))
    meta = dict(d=d, bs=wl["bs"], int8=wl["int8"], G=G)
    cores = os.cpu_count() or 1
    workers = min(cores, len(units))
    env_keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in env_keys}
    for k in env_keys:
        os.environ[k] = "1"
    try:
        ctx = mp.get_context("spawn")
        with ctx.Pool(workers, initializer=_pool_init, initargs=(ctx.Barrier(workers),)) as pool:
            t1, steps, b1, _ = pool.apply(_oracle_task, ((meta, units, max_steps, budget_s, False),))
            res = pool.map(_oracle_task, [(meta, units[i::workers], steps, None, True) for i in range(workers)],
                           chunksize=1)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    tn = max(r[0] for r in res)
    bn = sum(r[2] for r in res)
    tokens = nseq * steps / (wl["L"] * wl["repeat"])  # whole decode steps: all layers (and repeats)
    sample = (f"{steps} decode step(s) of layer 0 for {len(units)} (sequence, kv head) units "
              f"({nseq} sequence(s), contexts {min(ctxs[:nseq])}-{max(ctxs[:nseq])} tokens), every query head of "
              f"each unit's group; scaled per byte")
    return dict(single_gbs=b1 / t1 / 1e9, single_s=t1, all_gbs=bn / tn / 1e9, all_s=tn, workers=workers,
                cpu_count=cores, steps=steps, sample=sample, all_tokens_per_s=tokens / tn,
                single_tokens_per_s=tokens / t1)


def cpu_baseline_entry(r: dict) -> dict:
    """The bench line's cpu_baseline object from oracle_baseline's result."""
    return {"value": round(r["all_gbs"], 4), "unit": "GB/s", "cores": r["workers"], "kind": "oracle",
            "sample": r["sample"], "seconds": round(r["all_s"], 2),
            "tokens_per_s": round(r["all_tokens_per_s"], 3), "host_cpu_count": r["cpu_count"],
            "single_thread": {"value": round(r["single_gbs"], 4), "unit": "GB/s", "cores": 1,
                              "seconds": round(r["single_s"], 2),
                              "tokens_per_s": round(r["single_tokens_per_s"], 3)}}


# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--e2e-steps", type=int, default=40)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="tts_talker", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true", help="launch each kernel from Python instead of a CUDA graph")
    ap.add_argument("--split", type=int, default=None, help="split_tokens (default: sized to one wave)")
    ap.add_argument("--separate-merge", action="store_true", help="merge split-K partials in a second kernel")
    ap.add_argument("--no-pdl", action="store_true", help="launch kernels without programmatic dependent launch")
    ap.add_argument("--layers", type=int, default=None,
                    help="run the workload with this many layers (same per-layer launch; for small profiler "
                         "captures -- the line then names the layer count in config)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    wl = WORKLOADS[args.workload]
    if args.layers is not None:
        if args.layers < 1:
            ap.error("--layers must be >= 1")
        wl = dict(wl, L=args.layers)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    peak, peak_kind = _peaks()

    if args.impl == "reference":
        if rank != 0:
            return
        r = oracle_baseline(wl, budget_s=20.0)
        gbs, tps = r["all_gbs"], r["all_tokens_per_s"]
        line = {"impl": "reference", "metric": "paged decode-attention KV GB/s", "value": round(gbs, 4),
                "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (seeded counter-based generator)",
                "config": {"workload": args.workload, "desc": wl["desc"]},
                "tokens_per_s": round(tps, 3),
                "cpu_baseline": cpu_baseline_entry(r),
                "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    if world > 1:
        torch.distributed.init_process_group("nccl")
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    from paged_kv_cache_56_gb300 import build as _build
    _build.build()
    if args.workload == "trace":
        r = run_trace(args, wl)
        value = r["nbytes"] / (r["ms"] * 1e-3) / 1e9
        line = {"metric": "paged decode-attention KV GB/s", "value": round(value, 2), "unit": "GB/s",
                "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(r["ms"] / args.steps, 4), "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "int8 KV / bf16 q,out / fp32 accumulate",
                "data": "synthetic (seeded counter-based generator)",
                "config": {"workload": "trace", "desc": wl["desc"], "split_tokens": r["split"],
                           **({"layers": wl["L"]} if args.layers is not None else {}),
                           "timed": "decode kernels of each step (admission prefill excluded)",
                           "running_at_end": r["running"], "finished": r["finished"], "kv_pool_at_end": r["pool"]},
                "tokens_per_s": round(r["ntok"] / (r["ms"] * 1e-3), 1),
                "roofline": {"bound": "hbm", "achieved": round(value, 1), "peak": peak, "unit": "GB/s",
                             "frac": round(value / peak, 4), "traffic": None, "peak_kind": peak_kind},
                "clocks": r["clocks"], "gpu_launches": r["launches"], "e2e": None}
        print(json.dumps(line), flush=True)
        return
    r = run_device(args, wl, rank, world)
    if rank != 0:
        torch.distributed.destroy_process_group()
        return
    ms_step = r["ms"] / args.steps
    value = job_gbs(r["step_bytes"], world, r["ms"])
    attn_avg_ms = r["attn_call_ms"]
    achieved = r["attn_bytes"] / (attn_avg_ms * 1e-3) / 1e9
    line = {
        "metric": "paged decode-attention KV GB/s", "value": round(value, 2), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8 KV / bf16 q,out / fp32 accumulate" if wl["int8"] else "bf16 KV / fp32 accumulate",
        "data": "synthetic (seeded counter-based generator)",
        "config": {"workload": args.workload, "desc": wl["desc"], "split_tokens": r["split"],
                   **({"layers": wl["L"]} if args.layers is not None else {}),
                   "ctx_range": list(r["ctx"]), "l2": "inputs larger than L2 (per-step KV >> 129 MB)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "launch": "CUDA graph per step" if r["graph"] else "eager",
                   "split_merge": "separate kernel" if args.separate_merge else "fused (last split merges)",
                   "programmatic_dependent_launch": not args.no_pdl},
        "tokens_per_s": round(wl["B"] * world / (ms_step * 1e-3), 1),
        "hbm_frac_of_step": round(value / world / peak, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": measured_traffic(args.workload),
                     "peak_kind": peak_kind,
                     "kernel": "decode_kernel via pkv_decode_step (append + quantize-on-fill + attention + split-K merge)",
                     "bytes_per_launch": int(r["attn_bytes"]), "avg_launch_us": round(attn_avg_ms * 1e3, 2),
                     "timing": "CUDA events over back-to-back replays of the step's kernels"},
        "clocks": r["clocks"],
        "gpu_launches": r["launches"],
        "e2e": r["e2e"],
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_entry(oracle_baseline(wl, budget_s=10.0))
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
