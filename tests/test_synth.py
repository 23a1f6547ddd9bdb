"""The seeded input generator: deterministic, sliceable, roughly N(0,1)."""

import math

import torch

from paged_kv_cache_56_gb300 import synth


def test_rows_are_pure_functions_of_position():
    full = synth.kv_rows(3, 1, synth.KIND_K, 5, torch.arange(300), 4, 16)
    part = synth.kv_rows(3, 1, synth.KIND_K, 5, torch.tensor([7, 299, 0]), 4, 16)
    assert torch.equal(part, full[[7, 299, 0]])
    chunked = synth.kv_rows(3, 1, synth.KIND_K, 5, torch.arange(300), 4, 16, chunk_rows=17)
    assert torch.equal(chunked, full)
    multi = synth.kv_rows(3, 1, synth.KIND_K, torch.tensor([5, 6, 5]), torch.tensor([1, 1, 2]), 4, 16)
    other = synth.kv_rows(3, 1, synth.KIND_K, 6, torch.tensor([1]), 4, 16)
    assert torch.equal(multi[0], full[1]) and torch.equal(multi[2], full[2])
    assert torch.equal(multi[1], other[0]) and not torch.equal(multi[1], full[1])


def test_streams_differ():
    a = synth.kv_rows(3, 0, synth.KIND_K, 0, torch.arange(8), 2, 8)
    assert not torch.equal(a, synth.kv_rows(3, 0, synth.KIND_V, 0, torch.arange(8), 2, 8))
    assert not torch.equal(a, synth.kv_rows(3, 1, synth.KIND_K, 0, torch.arange(8), 2, 8))
    assert not torch.equal(a, synth.kv_rows(4, 0, synth.KIND_K, 0, torch.arange(8), 2, 8))
    q0 = synth.q_rows(3, 0, 0, [0, 1], 4, 8)
    assert not torch.equal(q0, synth.q_rows(3, 0, 1, [0, 1], 4, 8))
    assert not torch.equal(q0[0], q0[1])


def test_moments_and_multipliers():
    x = synth.kv_rows(11, 0, synth.KIND_V, 0, torch.arange(4096), 8, 128).float()
    assert abs(x.mean().item()) < 0.01 and abs(x.std().item() - 1) < 0.01
    assert x.abs().max().item() < 4.4
    m = synth.head_multipliers(11, 0, synth.KIND_K, 1000)
    assert m.min() >= 0.1 and m.max() <= 4.0 and abs(m.mean().item() - 2.05) < 0.1
    y = synth.kv_rows(11, 0, synth.KIND_V, 0, torch.arange(64), 8, 128, mult=m[:8]).float()
    base = synth.kv_rows(11, 0, synth.KIND_V, 0, torch.arange(64), 8, 128).float()
    ratio = (y / base.where(base != 0, torch.ones_like(base)))[base.abs() > 0.5]
    assert ratio.min() > 0.09 and ratio.max() < 4.1
    o = synth.outlier_multipliers(11, 0, synth.KIND_K, 64, 128)
    frac = (o == 20.0).float().mean().item()
    assert 0.005 < frac < 0.015 and set(o.unique().tolist()) == {1.0, 20.0}


def test_permutation_and_trace():
    p = synth.permutation(9, 1000)
    assert sorted(p) == list(range(1000)) and p != list(range(1000))
    assert p == synth.permutation(9, 1000)
    tr = synth.trace_requests(1234, 2000)
    assert abs(len(tr) / 2000 - 2.0) < 0.1
    prompts = [r[2] for r in tr]
    outs = [r[3] for r in tr]
    assert min(prompts) >= 16 and max(prompts) <= 4096
    med = sorted(prompts)[len(prompts) // 2]
    assert abs(math.log(med) - (math.log(16) + math.log(4096)) / 2) < 0.2  # log-uniform median
    assert min(outs) >= 1 and abs(sum(outs) / len(outs) - 300) < 20
