"""Decode attention over K and V of very different magnitudes, against the
oracle, through the C ABI.

The INT8 cache's scale is max|x| / 127 for any block, with no bound on its
size ("轻量级推理引擎实战：KV Cache 量化与连续批处理的底层优化" §3), so a
cache can hold V blocks with scales from ~1e-8 to ~1e36. The tests give each
kv head its own K and V magnitude (1e-4 .. 1e7), and let the V magnitude
change from block to block inside one sequence, for bf16 and INT8 caches,
with and without splits. Outputs are compared after dividing both sides by
the V magnitude, so that the absolute term of the tolerance cannot hide a
relative error, and must all be finite."""

import numpy as np
import pytest
import torch

from harness import ATOL, RTOL, Workload, assert_close
from libpkv import ensure_built
from oracle.attention import decode_attention
from paged_kv_cache_56_gb300 import synth

pytestmark = pytest.mark.gpu

MULTS = (1e-4, 1e-2, 1e4, 1e7)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _per_head(k_mult, v_mult):
    km = torch.tensor(k_mult, dtype=torch.float32)
    vm = torch.tensor(v_mult, dtype=torch.float32)

    def f(layer, kind, pos):
        m = vm if kind == synth.KIND_V else km
        return m[None, :].expand(pos.numel(), -1)
    return f


def _run(w: Workload, steps: int, v_div):
    """Decode `steps` steps; checks out / v_div against oracle / v_div.
    v_div: fp64 [Hq] divisor per query head."""
    for t in range(steps):
        out = w.step().float().cpu().numpy()
        assert np.isfinite(out).all(), f"step {t}: non-finite outputs"
        for i in range(w.B):
            ref = w.oracle_out(0, i, t)
            assert_close(out[0, i] / v_div[:, None], ref / v_div[:, None], f"step {t} seq {i}")
    assert w.error_bits() == 0


@pytest.mark.parametrize("int8", [False, True], ids=["bf16", "int8"])
@pytest.mark.parametrize("split", [0, 32])
@pytest.mark.parametrize("d", [64, 128])
def test_kv_heads_of_every_magnitude(int8, split, d):
    """Head h: V x MULTS[h], K x MULTS[3 - h] (large K: a near one-hot softmax;
    small K: a near-uniform one)."""
    hkv, g = 4, 2
    w = Workload(seed=31, num_layers=1, prior=(100, 47, 16, 3), Hq=hkv * g, Hkv=hkv, d=d, bs=16, num_blocks=64,
                 int8=int8, split_tokens=split, max_blocks=9,
                 kv_scale=_per_head(list(reversed(MULTS)), list(MULTS)))
    _run(w, 4, np.repeat(np.array(MULTS, dtype=np.float64), g))


@pytest.mark.parametrize("int8", [False, True], ids=["bf16", "int8"])
@pytest.mark.parametrize("split", [0, 64])
@pytest.mark.parametrize("favour_small", [False, True], ids=["flat_k", "small_v_blocks_win"])
def test_v_magnitude_changing_from_block_to_block(int8, split, favour_small):
    """Inside each sequence the V magnitude of block n is 10^((n % 9) - 4), so
    a warp meets V scales 1e8 apart in turn. favour_small: K x 3 on the blocks
    whose V magnitude is <= 1e-2, so that the softmax weight sits on the small
    V blocks while the large ones still contribute."""
    def f(layer, kind, pos):
        e = (pos // 16) % 9 - 4
        if kind == synth.KIND_V:
            m = torch.pow(torch.tensor(10.0), e.to(torch.float32))
        else:
            m = torch.where(e <= -2, torch.tensor(3.0), torch.tensor(1.0)) if favour_small else torch.ones(pos.numel())
        return m[:, None].expand(-1, 2)
    w = Workload(seed=32, num_layers=1, prior=(300, 257, 143, 9), Hq=8, Hkv=2, d=128, bs=16, num_blocks=96,
                 int8=int8, split_tokens=split, max_blocks=21, kv_scale=f)
    # The absolute term of the tolerance is taken relative to the magnitude of
    # the values each output averages, S = sum_t w_t |v_t| (oracle weights):
    # for V ~ N(0, 1) that is the plain tolerance (S ~ 0.8), and an output that
    # cancels to near zero inside a row of magnitude 1e3 is held to 2e-3 of
    # what it averages, not to 2e-3 absolute.
    for t in range(3):
        out = w.step().float().cpu().numpy()
        assert np.isfinite(out).all(), f"step {t}: non-finite outputs"
        for i in range(w.B):
            h = w.history(0, i, w.prior[i] + t + 1)
            k, v = h.context()
            q = w.q_for(0, t, [w.req_ids[i]], "cpu")[0].float().numpy()
            ref, wts = decode_attention(q, k, v, w.sm_scale, return_weights=True)
            g = w.Hq // w.Hkv
            mag = np.stack([wts[hq] @ np.abs(v[:, hq // g, :]) for hq in range(w.Hq)])
            err = np.abs(out[0, i] - ref)
            bad = err > ATOL * mag + RTOL * np.abs(ref)
            assert not bad.any(), (f"step {t} seq {i}: {bad.sum()} outside; worst excess "
                                   f"{np.max(err - ATOL * mag - RTOL * np.abs(ref)):.3g}")
    assert w.error_bits() == 0
