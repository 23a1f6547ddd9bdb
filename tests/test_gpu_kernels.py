"""GPU tests of single entry points: the split-K merge against the oracle's
merge of partial softmax states, zero-length contexts, device-side checks of
block ids / slots / context lengths, and quantization special cases."""

import math

import numpy as np
import pytest
import torch

from harness import assert_close
from libpkv import ensure_built
from oracle.attention import merge_partials
from oracle.quantize import quantize_block
from paged_kv_cache_56_gb300 import pkv
from paged_kv_cache_56_gb300.runtime import LayerCache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


@pytest.mark.parametrize("d", [64, 128])
def test_splitk_reduce_matches_oracle_merge(d):
    gen = torch.Generator().manual_seed(d)
    B, Hq, split, max_splits = 3, 4, 32, 9
    ctx = torch.tensor([1, 200, 288], dtype=torch.int32)
    ws_o = torch.randn(B, Hq, max_splits, d, generator=gen) * 3
    ws_ml = torch.empty(B, Hq, max_splits, 2)
    ws_ml[..., 0] = torch.randn(B, Hq, max_splits, generator=gen) * 20
    ws_ml[..., 1] = torch.rand(B, Hq, max_splits, generator=gen) * 50 + 0.5
    out = torch.empty(B, Hq, d, dtype=torch.bfloat16, device="cuda")
    pkv.pkv_splitk_reduce(ws_o.cuda().contiguous(), ws_ml.cuda().contiguous(), ctx.cuda(), Hq, d, split,
                          max_splits, out)
    got = out.float().cpu().numpy()
    for b in range(B):
        ns = -(-int(ctx[b]) // split)
        for h in range(Hq):
            ref = merge_partials(ws_ml[b, h, :ns, 0].numpy(), ws_ml[b, h, :ns, 1].numpy(), ws_o[b, h, :ns].numpy(),
                                 base=2.0)
            assert_close(got[b, h], ref, f"b{b} h{h}")


def _tiny_cache(int8, num_blocks=8):
    return LayerCache(num_blocks, 4, 2, 64, 16, int8, max_slots=2, device="cuda")


@pytest.mark.parametrize("int8", [False, True], ids=["bf16", "int8"])
@pytest.mark.parametrize("split", [0, 16])
def test_zero_length_context_gives_zero_row(int8, split):
    lc = _tiny_cache(int8)
    q = torch.randn(2, 4, 64, device="cuda").to(torch.bfloat16)
    tables = torch.tensor([[0, 1], [2, 3]], dtype=torch.int32, device="cuda")
    ctx = torch.tensor([0, 0], dtype=torch.int32, device="cuda")
    slots = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    out = torch.full((2, 4, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    ms = 2 if split else 0
    ws = dict(ws_o=torch.empty(2 * 4 * 2 * 64, device="cuda"), ws_ml=torch.empty(2 * 4 * 2 * 2, device="cuda"),
              ws_count=torch.zeros(4, dtype=torch.int32, device="cuda")) if split else {}
    pkv.pkv_decode_attention(lc.desc, q, tables, ctx, slots, 0.125, out, split, ms, **ws)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0
    assert lc.error_bits() == 0


def test_bad_table_entries_are_reported_and_skipped():
    lc = _tiny_cache(False)
    lc.k_pool.fill_(1.0)
    lc.v_pool.fill_(2.0)
    q = torch.ones(1, 4, 64, dtype=torch.bfloat16, device="cuda")
    tables = torch.tensor([[0, 99]], dtype=torch.int32, device="cuda")  # block 99 of 8
    ctx = torch.tensor([32], dtype=torch.int32, device="cuda")
    out = torch.empty(1, 4, 64, dtype=torch.bfloat16, device="cuda")
    pkv.pkv_decode_attention(lc.desc, q, tables, ctx, None, 0.125, out)
    torch.cuda.synchronize()
    assert lc.error_bits() & pkv.PKV_DEVERR_BLOCK_ID
    # the valid block still contributes: V == 2 everywhere there
    assert torch.allclose(out.float(), torch.full_like(out.float(), 2.0))
    # an out-of-range value in device memory reads back as PKV_ERR_INVALID
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_sync_status(lc.desc)
    assert e.value.code == pkv.PKV_ERR_INVALID
    assert pkv.pkv_sync_status(lc.desc, raise_on_error=False) == 0  # cleared
    ctx = torch.tensor([33], dtype=torch.int32, device="cuda")  # more than 2 blocks * 16
    pkv.pkv_decode_attention(lc.desc, q, torch.tensor([[0, 1]], dtype=torch.int32, device="cuda"), ctx, None,
                             0.125, out)
    torch.cuda.synchronize()
    assert lc.error_bits() & pkv.PKV_DEVERR_CTX_LEN


def test_bad_slots_and_offsets_are_reported():
    lc = _tiny_cache(True)
    rows = torch.ones(2, 2, 64, dtype=torch.bfloat16, device="cuda")
    pkv.pkv_append_kv(lc.desc, rows, rows, None, torch.tensor([0, 16], dtype=torch.int32, device="cuda"),
                      torch.tensor([5, 0], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    bits = lc.error_bits()
    assert bits & pkv.PKV_DEVERR_SLOT and bits & pkv.PKV_DEVERR_OFFSET
    assert torch.count_nonzero(lc.k_tail).item() == 0  # nothing was written
    lc.err.zero_()
    pkv.pkv_quantize_full_blocks(lc.desc, torch.tensor([-1, 3, 50], dtype=torch.int32, device="cuda"),
                                 torch.tensor([0, 9, 0], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    bits = lc.error_bits()
    assert bits & pkv.PKV_DEVERR_SLOT and bits & pkv.PKV_DEVERR_BLOCK_ID  # -1 is padding, not an error


def _quantize_on_gpu(x: np.ndarray):
    """x: [bs=16, d=64] bf16-valued; quantizes it as one (block, head) slab."""
    lc = LayerCache(2, 1, 1, 64, 16, True, max_slots=1, device="cuda")
    src = torch.from_numpy(x).to(torch.bfloat16).reshape(16, 1, 64).cuda()
    pkv.pkv_quantize_blocks_from(lc.desc, src, src, torch.tensor([1], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    return lc.k_pool[1, 0].cpu().numpy(), lc.scales[1, 0, 0].cpu().numpy()


@pytest.mark.parametrize("case", ["zero", "tiny", "single", "ties", "division_ties", "random", "outliers"])
def test_quantize_special_cases_bit_exact(case):
    gen = torch.Generator().manual_seed(3)
    x = np.zeros((16, 64), np.float32)
    if case == "tiny":
        x[3, 5] = 2.0 ** -21
        x[9, 1] = -(2.0 ** -20)
    elif case == "single":
        x[7, 7] = -3.0
    elif case == "ties":
        x.flat[:120] = [(k + 0.5) * 0.25 for k in range(-60, 60)]
        x.flat[500] = 127 * 0.25
    elif case == "division_ties":
        x.flat[:4] = [13.0, 6.5, -6.5, 0.0]
    elif case == "random":
        x = (torch.randn(16, 64, generator=gen) * 3).numpy()
    elif case == "outliers":
        x = torch.randn(16, 64, generator=gen).numpy()
        x[:, 11] *= 20
    x = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    q, s = _quantize_on_gpu(x)
    q_ref, s_ref = quantize_block(x)
    assert np.array_equal(q, q_ref)
    assert np.float32(s).view(np.uint32) == np.float32(s_ref).view(np.uint32)


@pytest.mark.parametrize("split", [0, 32])
def test_bounded_wait_runs_out_and_the_gpu_recovers(split):
    """A bulk copy that is never issued (the library's test hook) makes its
    bounded wait run out: the kernel reports PKV_DEVERR_TIMEOUT, drains its
    other copies and returns, and the next step on the same cache is right."""
    from harness import Workload
    w = Workload(seed=23, num_layers=1, prior=(100, 17, 33, 1), Hq=4, Hkv=2, d=64, bs=16, num_blocks=64, int8=True,
                 split_tokens=split, max_blocks=9)
    descs = [lc.desc for lc in w.cache.layers]
    pkv.pkv_debug_skip_copy(0)  # tile 0 of warp 0 of the first CTA: sequence 0 has pool tiles
    try:
        w.step()
        # the status call waits for the step, reads the error word and clears it
        with pytest.raises(pkv.PkvError) as e:
            pkv.pkv_sync_status(descs)
        assert e.value.code == pkv.PKV_ERR_DEVICE_TIMEOUT
    finally:
        pkv.pkv_debug_skip_copy(-1)
    assert w.error_bits() == 0
    assert pkv.pkv_sync_status(descs) == 0
    out = w.step().float().cpu().numpy()  # the cache itself was written by the append kernels
    for i in range(w.B):
        assert_close(out[0, i], w.oracle_out(0, i, 1), f"seq {i}")
    assert w.error_bits() == 0
