"""Decode over a work list (pkv_plan_segments + pkv_decode_layers_planned):
the (sequence, kv head) token runs of a step cut into equal pieces, one per
CTA, with pairs split across CTAs merged by the last to arrive. Against the
oracle element by element, pools byte for byte, for mixed context lengths
(empty, one token, block edges, long), bf16 and INT8 caches, 16- and 64-token
blocks, with the step's append and quantize-on-fill fused in, and with few
CTAs (many cuts per pair) and many."""

import numpy as np
import pytest
import torch

from harness import Workload, assert_close
from libpkv import ensure_built
from paged_kv_cache_56_gb300 import pkv, synth
from paged_kv_cache_56_gb300.runtime import StepBuffers

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _run(w: Workload, bufs: StepBuffers, t: int, fused: bool):
    plan = w.cache.plan_step(w.req_ids)
    bufs.upload(plan)
    L, B = w.L, w.B
    pos = torch.tensor(plan.positions, dtype=torch.int64)
    q = torch.stack([w.q(li, t, w.req_ids) for li in range(L)])
    k = torch.stack([w.kv(li, synth.KIND_K, w.req_ids, pos) for li in range(L)])
    v = torch.stack([w.kv(li, synth.KIND_V, w.req_ids, pos) for li in range(L)])
    if not fused:  # cache written first by the separate kernels, then attention only
        for li, lc in enumerate(w.cache.layers):
            pkv.pkv_append_kv(lc.desc, k[li], v[li], bufs.blk[:B], bufs.off[:B], bufs.slot[:B])
            if lc.int8:
                pkv.pkv_quantize_full_blocks(lc.desc, bufs.fill[:B], bufs.slot[:B])
        k = v = None
    out = torch.empty((L, B, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    pkv.pkv_decode_layers_planned(pkv.desc_array([lc.desc for lc in w.cache.layers]), q, k, v, bufs.tab[:B],
                                  bufs.ctx[:B], bufs.slot[:B], w.sm_scale, out, bufs.seg_plan, bufs.ws_o, bufs.ws_ml,
                                  bufs.ws_count)
    w.cache.commit_step(w.req_ids)
    return out


PRIOR = (0, 1, 15, 16, 17, 100, 400, 1000)


@pytest.mark.parametrize("ctas", [5, 64])
@pytest.mark.parametrize("fused", [True, False], ids=["fused_step", "attention_only"])
@pytest.mark.parametrize("int8,bs,d", [(True, 16, 128), (False, 16, 64), (True, 64, 128), (False, 64, 128)],
                         ids=["int8_bs16_d128", "bf16_bs16_d64", "int8_bs64_d128", "bf16_bs64_d128"])
def test_work_list_matches_oracle(int8, bs, d, fused, ctas):
    w = Workload(seed=60 + bs + d, num_layers=2, prior=PRIOR, Hq=8, Hkv=2, d=d, bs=bs, num_blocks=160, int8=int8,
                 split_tokens=0, max_blocks=-(-1100 // bs) + 1, fused_step=True)
    bufs = StepBuffers(w.cache, w.B, 0, fused_merge=True, work_list_ctas=ctas)
    for t in range(18):
        out = _run(w, bufs, t, fused).float().cpu().numpy()
        assert bufs.plan_info["ctas_used"] <= ctas
        if t in (0, 1, 17):
            for layer in range(2):
                for i in range(w.B):
                    assert_close(out[layer, i], w.oracle_out(layer, i, t), f"step {t} layer {layer} seq {i}")
    assert w.error_bits() == 0
    assert int(bufs.ws_count.abs().sum()) == 0  # counters left at zero
    for layer in range(2):
        for i in range(w.B):
            w.check_pool_bytes(layer, i, w.prior[i] + 18)


def test_work_list_agrees_with_uniform_split():
    """Same cache, same step: the work-list decode and the one-wave uniform
    split agree within the fp32 merge-order tolerance."""
    outs = {}
    for mode in ("split", "work_list"):
        w = Workload(seed=91, num_layers=1, prior=(3000, 5, 700, 64, 2222, 1), Hq=32, Hkv=8, d=128, bs=16,
                     num_blocks=480, int8=True, split_tokens=256, max_blocks=200, fused_step=True)
        if mode == "split":
            outs[mode] = w.step().float().cpu().numpy()
        else:
            bufs = StepBuffers(w.cache, w.B, 0, fused_merge=True, work_list_ctas=608)
            outs[mode] = _run(w, bufs, 0, True).float().cpu().numpy()
        assert w.error_bits() == 0
    ref = outs["split"]
    assert np.abs(outs["work_list"] - ref).max() <= 2e-3 + 1e-2 * np.abs(ref).max()


@pytest.mark.parametrize("int8", [False, True], ids=["bf16", "int8"])
def test_work_list_zero_context_rows(int8):
    """A sequence with no tokens gets one empty unit, whose output row is zero;
    the others are unaffected."""
    w = Workload(seed=5, num_layers=1, prior=(40, 90, 7), Hq=8, Hkv=2, d=64, bs=16, num_blocks=32, int8=int8,
                 max_blocks=8)
    bufs = StepBuffers(w.cache, w.B, 0, fused_merge=True, work_list_ctas=6)
    plan = w.cache.plan_step(w.req_ids)
    ctx = np.array(plan.ctx_lens) - 1  # attend over the prior tokens only (no append this call)
    ctx[1] = 0
    bufs.upload(plan)
    off, segs, info = pkv.pkv_plan_segments(ctx, 2, 16, 6, bufs.seg_cap)
    bufs.ctx[: w.B].copy_(torch.from_numpy(ctx.astype(np.int32)))
    bufs.segoff.copy_(torch.from_numpy(off))
    bufs.segs.copy_(torch.from_numpy(segs))
    sp = pkv.SegmentPlan(seg_offsets=bufs.segoff.data_ptr(), segs=bufs.segs.data_ptr(), num_ctas=6,
                         max_splits=bufs.max_splits, max_unit_tokens=info["max_unit_tokens"])
    q = w.q(0, 0, w.req_ids)[None]
    out = torch.full((1, w.B, 8, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    pkv.pkv_decode_layers_planned(pkv.desc_array([w.cache.layers[0].desc]), q, None, None, bufs.tab[: w.B],
                                  bufs.ctx[: w.B], bufs.slot[: w.B], w.sm_scale, out, sp, bufs.ws_o, bufs.ws_ml,
                                  bufs.ws_count)
    o = out[0].float().cpu().numpy()
    assert not o[1].any()
    from oracle.attention import decode_attention
    for i in (0, 2):
        k, v = w.history(0, i, int(ctx[i])).context()
        assert_close(o[i], decode_attention(w.q(0, 0, [w.req_ids[i]], "cpu")[0].float().numpy(), k, v, w.sm_scale),
                     f"seq {i}")
    assert w.error_bits() == 0
