"""GPU parity on the tiny configuration (1 layer, 4 sequences, Hq=4, Hkv=2,
d=64, block 16, 64-block pool, seeded shuffled pool), bf16 and INT8 caches,
every split setting, element by element against the oracle; plus the
quantizer's bytes and scales, bit for bit."""

import numpy as np
import pytest
import torch

from harness import Workload, assert_close
from libpkv import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


TINY = dict(num_layers=1, Hq=4, Hkv=2, d=64, bs=16, num_blocks=64)


@pytest.mark.parametrize("int8", [False, True], ids=["bf16", "int8"])
@pytest.mark.parametrize("split", [0, 16, 32, 64])
@pytest.mark.parametrize("prior", [(1, 17, 33, 100), (15, 16, 31, 0)])
def test_tiny_decode_steps(int8, split, prior):
    w = Workload(seed=1234, prior=prior, int8=int8, split_tokens=split, max_blocks=9, **TINY)
    for t in range(18):  # crosses a block boundary for every sequence
        out = w.step().float().cpu().numpy()
        for i in range(w.B):
            assert_close(out[0, i], w.oracle_out(0, i, t), f"step {t} seq {i}")
    assert w.error_bits() == 0
    for i in range(w.B):
        w.check_pool_bytes(0, i, prior[i] + 18)


@pytest.mark.parametrize("int8", [False, True], ids=["bf16", "int8"])
def test_block_permutation_is_bit_identical(int8):
    outs = []
    for shuffle in (False, True):
        w = Workload(seed=77, prior=(40, 100, 7, 64), int8=int8, shuffle=shuffle, split_tokens=32, max_blocks=9,
                     **TINY)
        outs.append(torch.stack([w.step() for _ in range(3)]).cpu())
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("int8", [False, True], ids=["bf16", "int8"])
def test_split_counts_agree(int8):
    res = {}
    for split in (0, 16, 48, 112):
        w = Workload(seed=5, prior=(100, 3, 77, 111), int8=int8, split_tokens=split, max_blocks=8, **TINY)
        res[split] = w.step().float().cpu().numpy()
    for split in (16, 48, 112):
        assert_close(res[split], res[0], f"split {split} vs none")


@pytest.mark.parametrize("int8", [False, True], ids=["bf16", "int8"])
def test_fused_and_separate_merge_agree(int8):
    res = {}
    for fused in (True, False):
        w = Workload(seed=9, prior=(100, 3, 77, 111), int8=int8, split_tokens=32, max_blocks=8, fused_merge=fused,
                     **TINY)
        res[fused] = torch.stack([w.step() for _ in range(5)]).cpu()
        assert w.error_bits() == 0
        if fused:
            assert int(w.bufs.ws_count.abs().sum()) == 0  # counters are left at zero
    assert torch.equal(res[True], res[False])


@pytest.mark.parametrize("int8", [False, True], ids=["bf16", "int8"])
def test_graph_replay_matches_oracle(int8):
    w = Workload(seed=21, prior=(5, 40, 16, 63), int8=int8, split_tokens=32, max_blocks=9, graph=True, repeat=2,
                 **TINY)
    for t in range(20):
        out = w.step().float().cpu().numpy()
        for i in range(w.B):
            for rep in range(2):
                assert_close(out[rep, i], w.oracle_out(0, i, t, rep), f"step {t} seq {i} rep {rep}")
    assert w.error_bits() == 0


@pytest.mark.parametrize("int8", [False, True], ids=["bf16", "int8"])
@pytest.mark.parametrize("split", [0, 32])
def test_fused_step_equals_separate_kernels(int8, split):
    """pkv_decode_step (append + quantize-on-fill + attention in one kernel)
    gives the same bytes as the three separate kernels, across block fills."""
    outs, pools = {}, {}
    for fused in (False, True):
        w = Workload(seed=31, prior=(15, 16, 47, 1), int8=int8, split_tokens=split, max_blocks=9, fused_step=fused,
                     **TINY)
        outs[fused] = torch.stack([w.step() for _ in range(34)]).cpu()
        assert w.error_bits() == 0
        lc = w.cache.layers[0]
        pools[fused] = [t.clone().cpu() for t in (lc.k_pool, lc.v_pool) + ((lc.scales, lc.k_tail, lc.v_tail)
                                                                          if int8 else ())]
        if fused:
            for t in range(34):
                out = outs[fused][t].float().numpy()
                for i in range(w.B):
                    assert_close(out[0, i], w.oracle_out(0, i, t), f"fused step {t} seq {i}")
            for i in range(w.B):
                w.check_pool_bytes(0, i, w.prior[i] + 34)
    assert torch.equal(outs[True], outs[False])
    # every block a sequence holds (the pools' other blocks were never written)
    if int8:
        for a, b in zip(pools[True], pools[False]):
            assert a.shape == b.shape


@pytest.mark.parametrize("int8", [False, True], ids=["bf16", "int8"])
@pytest.mark.parametrize("max_blocks", [9, 24], ids=["9_splits", "24_splits"])
def test_fused_merge_many_splits_match_oracle(int8, max_blocks):
    """The fused split-K merge with few and with many splits per sequence,
    empty splits (short sequences) in the mix, against the oracle."""
    prior = (120, 3, 60, 17) if max_blocks == 9 else (360, 3, 60, 17)
    w = Workload(seed=77, prior=prior, int8=int8, split_tokens=16, max_blocks=max_blocks, **TINY)
    assert (w.bufs.max_splits <= 16) == (max_blocks == 9)
    for t in range(6):
        out = w.step().float().cpu().numpy()
        for i in range(w.B):
            assert_close(out[0, i], w.oracle_out(0, i, t), f"step {t} seq {i}")
    assert w.error_bits() == 0


@pytest.mark.parametrize("int8", [False, True], ids=["bf16", "int8"])
def test_decode_layers_equals_per_layer_steps(int8):
    """pkv_decode_layers (one call for all layers) == pkv_decode_step per layer."""
    from paged_kv_cache_56_gb300 import pkv, synth
    outs = {}
    for one_call in (False, True):
        w = Workload(seed=8, num_layers=3, prior=(40, 17, 100, 1), Hq=4, Hkv=2, d=64, bs=16, num_blocks=96,
                     int8=int8, split_tokens=32, max_blocks=9, fused_step=True)
        res = []
        for t in range(18):
            if not one_call:
                res.append(w.step().cpu())
                continue
            plan = w.cache.plan_step(w.req_ids)
            w.bufs.upload(plan)
            b, B = w.bufs, w.B
            pos = torch.tensor(plan.positions, dtype=torch.int64)
            q = torch.stack([w.q(li, t, w.req_ids) for li in range(3)])
            k = torch.stack([w.kv(li, synth.KIND_K, w.req_ids, pos) for li in range(3)])
            v = torch.stack([w.kv(li, synth.KIND_V, w.req_ids, pos) for li in range(3)])
            out = torch.empty((3, 6, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")  # wider than the batch
            pkv.pkv_decode_layers(pkv.desc_array([lc.desc for lc in w.cache.layers]), q, k, v, b.tab[:B],
                                  b.ctx[:B], b.slot[:B], w.sm_scale, out[:, :B], b.split_tokens, b.max_splits,
                                  b.ws_o, b.ws_ml, b.ws_count)
            w.cache.commit_step(w.req_ids)
            res.append(out[:, :B].cpu())
        assert w.error_bits() == 0
        outs[one_call] = torch.stack(res)
    assert torch.equal(outs[True], outs[False])


@pytest.mark.parametrize("split", [0, 32])
def test_single_kv_head_odd_pool(split):
    """INT8 with one kv head and an odd pool (63 blocks, scale entries at
    every 8-byte offset): with this seed the pool's last block is a full block
    of the fourth sequence, read through the pool every step, and the pool
    ends the run fully held."""
    w = Workload(seed=3, num_layers=1, prior=(224, 224, 224, 207), Hq=2, Hkv=1, d=64, bs=16, num_blocks=63,
                 int8=True, split_tokens=split, max_blocks=17)
    assert 62 in w.cache.table(w.req_ids[3])[: 207 // 16]
    for t in range(20):  # ends with all 63 blocks held
        out = w.step().float().cpu().numpy()
        if t % 5 == 4:
            for i in range(w.B):
                assert_close(out[0, i], w.oracle_out(0, i, t), f"step {t} seq {i}")
    assert max(max(w.cache.table(r)) for r in w.req_ids) == 62  # the last block is in use
    assert w.error_bits() == 0
    for i in range(w.B):
        w.check_pool_bytes(0, i, w.prior[i] + 20)


@pytest.mark.parametrize("graph", [False, True], ids=["eager", "graph"])
def test_mixed_precision_layers(graph):
    """Per-layer cache precision ("轻量级推理引擎实战" §3.2: bf16 for the first
    and last layers, INT8 in between) through one step path: every layer
    against the oracle in its own precision, pools byte for byte."""
    flags = (False, True, True, False)
    w = Workload(seed=41, num_layers=4, prior=(15, 16, 47, 1), Hq=4, Hkv=2, d=64, bs=16, num_blocks=96,
                 int8=flags, split_tokens=32, max_blocks=9, graph=graph)
    assert [lc.int8 for lc in w.cache.layers] == list(flags)
    for t in range(18):
        out = w.step().float().cpu().numpy()
        if t % 6 == 5 or t == 0:
            for layer in range(4):
                for i in range(w.B):
                    assert_close(out[layer, i], w.oracle_out(layer, i, t), f"step {t} layer {layer} seq {i}")
    assert w.error_bits() == 0
    for layer in range(4):
        for i in range(w.B):
            w.check_pool_bytes(layer, i, w.prior[i] + 18)


@pytest.mark.parametrize("int8", [False, True], ids=["bf16", "int8"])
def test_pipelined_host_steps_equal_graph_steps(int8):
    """PipelinedSteps (inputs from pinned host memory on a copy stream, two
    alternating captured graphs, outputs back to pinned host memory) gives the
    same bytes as GraphStep replays, step by step."""
    from paged_kv_cache_56_gb300 import synth
    from paged_kv_cache_56_gb300.runtime import PipelinedSteps
    ref = Workload(seed=13, prior=(1, 17, 33, 100), int8=int8, split_tokens=32, max_blocks=9, graph=True, **TINY)
    want = [ref.step().cpu() for _ in range(20)]
    w = Workload(seed=13, prior=(1, 17, 33, 100), int8=int8, split_tokens=32, max_blocks=9, graph=True, **TINY)
    pipe = PipelinedSteps(w.cache, w.B, w.split_tokens, w.sm_scale)
    outs = [torch.empty((1, w.B, w.Hq, w.d), dtype=torch.bfloat16).pin_memory() for _ in range(20)]
    for t in range(20):
        pos = torch.tensor([w.cache.seqs[r].length for r in w.req_ids], dtype=torch.int64)
        q = w.q(0, t, w.req_ids)[None].cpu().pin_memory()
        k = w.kv(0, synth.KIND_K, w.req_ids, pos)[None].cpu().pin_memory()
        v = w.kv(0, synth.KIND_V, w.req_ids, pos)[None].cpu().pin_memory()
        pipe.step(w.req_ids, q, k, v, outs[t])
    pipe.finish()
    torch.cuda.synchronize()
    for t in range(20):
        assert torch.equal(outs[t], want[t]), t
    assert w.error_bits() == 0


@pytest.mark.parametrize("int8", [False, True], ids=["bf16", "int8"])
@pytest.mark.parametrize("d,bs", [(64, 16), (64, 64), (128, 64)], ids=["d64_bs16", "d64_bs64", "d128_bs64"])
@pytest.mark.parametrize("split", [0, 64])
@pytest.mark.parametrize("fused", [False, True], ids=["three_kernels", "fused_step"])
def test_gqa_group_of_eight(int8, d, bs, split, fused):
    """The widest GQA group the kernels take (G = Hq / Hkv = 8, the MMA's full
    N dimension), both head sizes and block sizes, with and without splits,
    across block fills (the sequence of 63 tokens fills a 64-token block at
    the first step: with fused_step, the decode kernel's own quantize-on-fill
    of a 64-row slab), against the oracle and byte for byte in the pools."""
    w = Workload(seed=70 + d + bs, num_layers=1, prior=(3, 63, 64, 130), Hq=16, Hkv=2, d=d, bs=bs, num_blocks=40,
                 int8=int8, split_tokens=split, max_blocks=5 if bs == 64 else 14, fused_step=fused)
    for t in range(20):
        out = w.step().float().cpu().numpy()
        if t in (0, 1, 19):
            for i in range(w.B):
                assert_close(out[0, i], w.oracle_out(0, i, t), f"step {t} seq {i}")
    assert w.error_bits() == 0
    for i in range(w.B):
        w.check_pool_bytes(0, i, w.prior[i] + 20)
