"""pkv_decode_attention_static_ws: decode attention for callers that cannot
allocate device memory while they decode (an engine that gives all free HBM to
its cache pool at start-up and forbids later allocations, code running inside
such an engine, a latency-critical loop that must not pay for cudaMalloc's
implicit synchronisation). Its split-K scratch is a fixed array inside the
library. Two calls in a row, through the C ABI, must agree with the oracle and
with the regular entry point (which uses a workspace the caller allocated),
and a warmed-up call must leave the device's free memory unchanged."""

import numpy as np
import pytest
import torch

from harness import Workload, assert_close
from libpkv import ensure_built
from paged_kv_cache_56_gb300 import pkv, synth

pytestmark = pytest.mark.gpu

CASES = {
    "tiny_int8": dict(num_layers=1, prior=(1, 17, 33, 100), Hq=4, Hkv=2, d=64, bs=16, num_blocks=64, int8=True,
                      split_tokens=32, max_blocks=9),
    "tiny_bf16": dict(num_layers=1, prior=(15, 16, 31, 0), Hq=4, Hkv=2, d=64, bs=16, num_blocks=64, int8=False,
                      split_tokens=16, max_blocks=9),
    "gqa_int8_2000": dict(num_layers=1, prior=(2000, 1999, 1500, 2047), Hq=16, Hkv=8, d=128, bs=16,
                          num_blocks=600, int8=True, split_tokens=128, max_blocks=130, head_scale=True),
    "tiny_int8_no_split": dict(num_layers=1, prior=(1, 17, 33, 100), Hq=4, Hkv=2, d=64, bs=16, num_blocks=64,
                               int8=True, split_tokens=0, max_blocks=9),
}


def _step_inputs(w: Workload):
    """Writes decode step 0's rows into the cache (regular kernels) and returns
    the query; the control arrays are in w.bufs."""
    c, bufs, lc = w.cache, w.bufs, w.cache.layers[0]
    plan = c.plan_step(w.req_ids)
    bufs.upload(plan)
    B = w.B
    pos = torch.tensor(plan.positions, dtype=torch.int64)
    pkv.pkv_append_kv(lc.desc, w.kv(0, synth.KIND_K, w.req_ids, pos), w.kv(0, synth.KIND_V, w.req_ids, pos),
                      bufs.blk[:B], bufs.off[:B], bufs.slot[:B])
    if c.int8:
        pkv.pkv_quantize_full_blocks(lc.desc, bufs.fill[:B], bufs.slot[:B])
    return w.q(0, 0, w.req_ids)


@pytest.mark.parametrize("name", sorted(CASES))
def test_static_ws_matches_oracle_and_regular_entry_point(name):
    ensure_built()
    w = Workload(seed=4321, **CASES[name])
    bufs, lc, B = w.bufs, w.cache.layers[0], w.B
    q = _step_inputs(w)
    oracle = np.stack([w.oracle_out(0, i, 0) for i in range(B)])
    regular = torch.empty((B, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    pkv.pkv_decode_attention(lc.desc, q, bufs.tab[:B], bufs.ctx[:B], bufs.slot[:B], w.sm_scale, regular,
                             bufs.split_tokens, bufs.max_splits, bufs.ws_o, bufs.ws_ml, bufs.ws_count)
    regular = regular.float().cpu().numpy()
    assert_close(regular, oracle, f"{name} regular entry point")
    outs = [torch.full((B, w.Hq, w.d), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    for call in range(2):
        free_before = torch.cuda.mem_get_info()[0]
        pkv.pkv_decode_attention_static_ws(lc.desc, q, bufs.tab[:B], bufs.ctx[:B], bufs.slot[:B], w.sm_scale,
                                           outs[call], bufs.split_tokens, bufs.max_splits)
        torch.cuda.synchronize()
        if call == 1:  # warmed up: the call itself takes no device memory
            assert torch.cuda.mem_get_info()[0] == free_before
        got = outs[call].float().cpu().numpy()
        assert_close(got, oracle, f"{name} call {call + 1} vs oracle")
        assert_close(got, regular, f"{name} call {call + 1} vs regular entry point")
    assert w.error_bits() == 0


def test_static_ws_rejects_requests_beyond_its_size_and_negative_splits():
    ensure_built()
    w = Workload(seed=1, **CASES["tiny_int8"])
    lc, bufs = w.cache.layers[0], w.bufs
    B, max_blocks = w.B, 4096
    tab = torch.full((B, max_blocks), -1, dtype=torch.int32, device="cuda")
    out = torch.empty((B, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    q = w.q(0, 0, w.req_ids)
    # 4096 splits x 4 sequences x 4 heads x (64 + 2) floats is more than the fixed array holds
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode_attention_static_ws(lc.desc, q, tab, bufs.ctx[:B], bufs.slot[:B], w.sm_scale, out, 16, 4096)
    assert e.value.code == pkv.PKV_ERR_TOO_LARGE
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode_attention_static_ws(lc.desc, q, bufs.tab[:B], bufs.ctx[:B], bufs.slot[:B], w.sm_scale, out,
                                           -16, 4)
    assert e.value.code == pkv.PKV_ERR_INVALID
