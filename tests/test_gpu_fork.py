"""Copy-on-write forking on the GPU ("vLLM核心概念" §3.2: requests that share
a prefix point at the same physical blocks, which are copied only when one of
them writes into a shared block -- parallel sampling from one prompt).

A parent with a 37-token prompt (two full blocks and a partly filled third)
is forked into two children; all three then decode their own tokens. Each
output is compared with the oracle's attention over that request's own
history (the parent's 37 prompt rows, then its own rows), the pools byte for
byte with the oracle's quantized histories, and the block tables with the
oracle allocator's copy-on-write semantics (shared full blocks stay shared,
the partly filled one is replaced for all but its last holder)."""

import math

import numpy as np
import pytest
import torch

from harness import assert_close
from libpkv import ensure_built
from oracle.attention import decode_attention
from oracle.cache import SequenceHistory
from paged_kv_cache_56_gb300 import pkv, synth
from paged_kv_cache_56_gb300.runtime import PagedKVCache, StepBuffers, decode_step, prefill

pytestmark = pytest.mark.gpu

SEED, L, HQ, HKV, D, BS, POOL = 17, 2, 4, 2, 64, 16, 64
PARENT, CHILDREN, PROMPT = 100, (101, 102), 37


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()
    pkv.pkv_set_programmatic_launch(False)


def _rows(layer, kind, req, lo, hi, device="cuda"):
    """K or V rows of request req at positions lo..hi-1: the parent's prompt
    rows below PROMPT, the request's own rows from PROMPT on."""
    pos = torch.arange(lo, hi)
    seqs = torch.where(pos < PROMPT, torch.full_like(pos, PARENT), torch.full_like(pos, req))
    return synth.kv_rows(SEED, layer, kind, seqs, pos, HKV, D, device=device)


def _history(layer, req, n, int8):
    h = SequenceHistory(HKV, D, BS, int8)
    h.append(_rows(layer, synth.KIND_K, req, 0, n, "cpu").float().numpy(),
             _rows(layer, synth.KIND_V, req, 0, n, "cpu").float().numpy())
    return h


def _check_pools(cache, req, n, int8):
    tab = cache.table(req)
    for layer in range(L):
        h = _history(layer, req, n, int8)
        lc = cache.layers[layer]
        if int8:
            for bi in range(n // BS):
                qk, sk, qv, sv = h.blocks[bi]
                b = tab[bi]
                assert np.array_equal(lc.k_pool[b].cpu().numpy(), qk), (req, layer, bi)
                assert np.array_equal(lc.v_pool[b].cpu().numpy(), qv), (req, layer, bi)
                sc = lc.scales[b].cpu().numpy()
                assert np.array_equal(sc[:, 0].view(np.uint32), sk.view(np.uint32))
                assert np.array_equal(sc[:, 1].view(np.uint32), sv.view(np.uint32))
        else:
            kr, vr = h.raw()
            for bi in range(-(-n // BS)):
                lo, hi = bi * BS, min(n, (bi + 1) * BS)
                b = tab[bi]
                assert np.array_equal(lc.k_pool[b, :, : hi - lo].float().cpu().numpy(),
                                      kr[lo:hi].transpose(1, 0, 2)), (req, layer, bi)
                assert np.array_equal(lc.v_pool[b, :, : hi - lo].float().cpu().numpy(),
                                      vr[lo:hi].transpose(1, 0, 2)), (req, layer, bi)


@pytest.mark.parametrize("split", [0, 32])
@pytest.mark.parametrize("int8", [False, True], ids=["bf16", "int8"])
def test_fork_parallel_sampling(int8, split):
    cache = PagedKVCache(L, POOL, HQ, HKV, D, BS, int8, max_slots=4, max_blocks_per_seq=8,
                         initial_order=synth.permutation(SEED, POOL))
    try:
        cache.add_sequence(PARENT, -(-PROMPT // BS))
        for layer in range(L):
            prefill(cache, layer, [PARENT], [_rows(layer, synth.KIND_K, PARENT, 0, PROMPT)],
                    [_rows(layer, synth.KIND_V, PARENT, 0, PROMPT)])
        cache.seqs[PARENT].length = PROMPT
        for c in CHILDREN:
            cache.fork(PARENT, c)
        reqs = [PARENT, *CHILDREN]
        t0 = cache.table(PARENT)
        assert all(cache.table(c) == t0 for c in CHILDREN)
        assert [pkv.pkv_block_refs(cache.alloc, b) for b in t0] == [3, 3, 3]
        free0 = pkv.pkv_num_free(cache.alloc)

        bufs = StepBuffers(cache, len(reqs), split)
        sm = 1.0 / math.sqrt(D)
        for t in range(30):  # positions 37..66: fills blocks 2 and 3, opens 4
            n = PROMPT + t
            q = [synth.q_rows(SEED, layer, t, reqs, HQ, D, device="cuda") for layer in range(L)]
            k = [torch.cat([_rows(layer, synth.KIND_K, r, n, n + 1) for r in reqs]) for layer in range(L)]
            v = [torch.cat([_rows(layer, synth.KIND_V, r, n, n + 1) for r in reqs]) for layer in range(L)]
            out = [torch.empty((len(reqs), HQ, D), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
            plan = decode_step(cache, bufs, reqs, q, k, v, out, sm)
            if t == 0:
                # the write into the shared partly filled block: private copies for
                # the first two holders, the last keeps the original
                assert len(plan.cow) == 2 and all(a == t0[2] for a, _ in plan.cow)
                tabs = [cache.table(r) for r in reqs]
                assert all(tb[:2] == t0[:2] for tb in tabs)
                assert len({tb[2] for tb in tabs}) == 3 and tabs[2][2] == t0[2]
                assert pkv.pkv_num_free(cache.alloc) == free0 - 2
            else:
                assert not plan.cow
            for layer in range(L):
                o = out[layer].float().cpu().numpy()
                for i, r in enumerate(reqs):
                    kk, vv = _history(layer, r, n + 1, int8).context()
                    qq = synth.q_rows(SEED, layer, t, [r], HQ, D)[0].float().numpy()
                    assert_close(o[i], decode_attention(qq, kk, vv, sm), f"step {t} req {r} layer {layer}")
        assert sum(lc.error_bits() for lc in cache.layers) == 0
        for r in reqs:
            _check_pools(cache, r, PROMPT + 30, int8)
        # the shared prompt blocks outlive the parent
        cache.remove_sequence(PARENT)
        assert [pkv.pkv_block_refs(cache.alloc, b) for b in t0[:2]] == [2, 2]
        for c in CHILDREN:
            cache.remove_sequence(c)
        assert pkv.pkv_num_free(cache.alloc) == POOL
    finally:
        cache.close()


@pytest.mark.parametrize("int8", [False, True], ids=["bf16", "int8"])
def test_copy_blocks_and_slots_bit_exact(int8):
    g = torch.Generator(device="cuda").manual_seed(5)
    cache = PagedKVCache(1, 16, HQ, HKV, D, BS, int8, max_slots=4, max_blocks_per_seq=4)
    try:
        lc = cache.layers[0]
        for t in (lc.k_pool, lc.v_pool) + ((lc.scales, lc.k_tail, lc.v_tail) if int8 else ()):
            t.view(torch.uint8).copy_(torch.randint(0, 256, t.view(torch.uint8).shape, generator=g,
                                                    device="cuda", dtype=torch.uint8))
        before = [t.clone() for t in (lc.k_pool, lc.v_pool) + ((lc.scales, lc.k_tail, lc.v_tail) if int8 else ())]
        src = torch.tensor([3, -1, 7, 9, 5], dtype=torch.int32, device="cuda")
        dst = torch.tensor([11, 2, 7, 16, 0], dtype=torch.int32, device="cuda")  # -1: skip; 7->7: skip; 16: bad
        pkv.pkv_copy_blocks(lc.desc, src, dst)
        torch.cuda.synchronize()
        assert lc.error_bits() == pkv.PKV_DEVERR_BLOCK_ID
        want = [t.clone() for t in before]
        for s, d in ((3, 11), (5, 0)):
            for w in want[: 3 if int8 else 2]:
                w[d] = w[s]
        for got, w in zip((lc.k_pool, lc.v_pool) + ((lc.scales,) if int8 else ()), want):
            assert torch.equal(got.view(torch.uint8), w.view(torch.uint8))
        if int8:
            lc.err.zero_()
            pkv.pkv_copy_slots(lc.desc, torch.tensor([2, 0], dtype=torch.int32, device="cuda"),
                               torch.tensor([1, 4], dtype=torch.int32, device="cuda"))
            torch.cuda.synchronize()
            assert lc.error_bits() == pkv.PKV_DEVERR_SLOT
            for got, w in zip((lc.k_tail, lc.v_tail), want[3:]):
                w[1] = w[2]
                assert torch.equal(got.view(torch.uint8), w.view(torch.uint8))
    finally:
        cache.close()
