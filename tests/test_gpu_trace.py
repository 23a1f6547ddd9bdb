"""The continuous-batching trace (200 decode steps, up to 128 running
requests, Hq=32, Hkv=8, d=128, 16-token blocks, INT8 cache, 32 layers, a
200-token shared prefix), in the launch configuration the benchmark times
(its split length, programmatic dependent launch, the driver's batch order):
sampled outputs against the oracle every 20th step, block conservation every
step, and the pools of sampled requests byte for byte at the end."""

import gc
import math

import numpy as np
import pytest
import torch

from harness import assert_close
from libpkv import ensure_built
from oracle.attention import decode_attention
from oracle.cache import SequenceHistory
from paged_kv_cache_56_gb300 import pkv, synth
from paged_kv_cache_56_gb300.runtime import PagedKVCache
from paged_kv_cache_56_gb300.trace import PREFIX_SEQ, TRACE_PDL, TRACE_SPLIT_TOKENS, TraceDriver

pytestmark = pytest.mark.gpu

SEED, STEPS, L, HQ, HKV, D, BS, POOL = 4242, 200, 32, 32, 8, 128, 16, 8192


def _history(drv: TraceDriver, layer: int, rid: int, n: int) -> SequenceHistory:
    h = SequenceHistory(HKV, D, BS, True)
    pos = torch.arange(n)
    h.append(drv.rows(layer, synth.KIND_K, rid, pos, "cpu").float().numpy(),
             drv.rows(layer, synth.KIND_V, rid, pos, "cpu").float().numpy())
    return h


@pytest.fixture(scope="module")
def run():
    ensure_built()
    pkv.pkv_set_programmatic_launch(TRACE_PDL)
    max_blocks = -(-(200 + 4096 + STEPS + 16) // BS)
    cache = PagedKVCache(L, POOL, HQ, HKV, D, BS, True, max_slots=129, max_blocks_per_seq=max_blocks,
                         initial_order=synth.permutation(SEED, POOL))
    drv = TraceDriver(cache, SEED, STEPS, max_running=128, split_tokens=TRACE_SPLIT_TOKENS)
    yield drv
    pkv.pkv_set_programmatic_launch(False)
    cache.close()
    del drv, cache
    gc.collect()
    torch.cuda.empty_cache()


def test_trace_matches_oracle(run):
    drv = run
    c = drv.cache
    checked = 0
    peak = 0
    rng = np.random.default_rng(7)
    for step in range(STEPS):
        rids, plan = drv.step()
        # every block is either free or held: private blocks + the shared prefix
        held = sum(len(c.table(r)) - len(drv.prefix_ids) for r in c.seqs if r != PREFIX_SEQ)
        assert pkv.pkv_num_free(c.alloc) + held + len(drv.prefix_ids) == POOL
        peak = max(peak, len(rids))
        if step % 20 == 19 and rids:
            out = drv.out[:, : len(rids)].float().cpu().numpy()
            for i in rng.choice(len(rids), size=min(2, len(rids)), replace=False):
                rid, ctx = rids[i], int(plan.ctx_lens[i])
                for layer in (0, L - 1):
                    h = _history(drv, layer, rid, ctx)
                    k, v = h.context()
                    q = drv.q_rows(layer, [rid], drv.step_no - 1, "cpu")[0].float().numpy()
                    ref = decode_attention(q, k, v, 1.0 / math.sqrt(D))
                    assert_close(out[layer, i], ref, f"step {step} rid {rid} layer {layer} ctx {ctx}")
                    checked += 1
    assert sum(lc.error_bits() for lc in c.layers) == 0
    assert checked >= 20
    assert peak > 32 and drv.finished  # the trace did fill up and requests did finish


def test_trace_pools_byte_exact(run):
    drv = run
    c = drv.cache
    running = [r for r in drv.running][:3]
    assert running
    for r in running:
        n = c.seqs[r.rid].length
        tab = c.table(r.rid)
        nf = n // BS
        for layer in (0, L - 1):
            h = _history(drv, layer, r.rid, n)
            lc = c.layers[layer]
            ids = torch.tensor(tab[:nf], dtype=torch.long, device="cuda")
            kp, vp, sc = lc.k_pool[ids].cpu().numpy(), lc.v_pool[ids].cpu().numpy(), lc.scales[ids].cpu().numpy()
            for bi in range(nf):
                qk, sk, qv, sv = h.blocks[bi]
                assert np.array_equal(kp[bi], qk) and np.array_equal(vp[bi], qv), (r.rid, layer, bi)
                assert np.array_equal(sc[bi, :, 0].view(np.uint32), sk.view(np.uint32))
                assert np.array_equal(sc[bi, :, 1].view(np.uint32), sv.view(np.uint32))
    # the shared prefix blocks are referenced by every running request
    for r in drv.running:
        assert c.table(r.rid)[: len(drv.prefix_ids)] == drv.prefix_ids
