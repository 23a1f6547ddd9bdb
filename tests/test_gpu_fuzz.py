"""Seeded random shapes against the oracle: GQA groups 1-8, head sizes 64
and 128, 16- and 64-token blocks, bf16 and INT8 caches, ragged contexts
(empty, one token, block edges, long), no split / small / large splits, a few
decode steps each, fused step or separate kernels, graph or eager -- every
output element against the fp64 oracle, INT8 pools byte for byte."""

import random

import pytest

from harness import Workload, assert_close
from libpkv import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_built()


def _case(i):
    rng = random.Random(1000 + i)
    g = rng.choice([1, 2, 4, 8])
    hkv = rng.choice([1, 2, 3])
    d = rng.choice([64, 128])
    bs = rng.choice([16, 64])
    int8 = rng.random() < 0.5
    B = rng.randint(1, 5)
    prior = [rng.choice([0, 1, bs - 1, bs, bs + 1, rng.randint(2, 600)]) for _ in range(B)]
    steps = rng.randint(1, 6)
    max_blocks = -(-(max(prior) + steps + 1) // bs) + rng.randint(0, 2)
    split = rng.choice([0, bs, 4 * bs, 16 * bs]) if rng.random() < 0.7 else 0
    if split and split % 16:
        split = 0
    fused = rng.random() < 0.5
    graph = fused and rng.random() < 0.5
    blocks = sum(-(-(p + steps) // bs) for p in prior) + rng.randint(0, 8)
    return dict(seed=2000 + i, num_layers=1, prior=tuple(prior), Hq=g * hkv, Hkv=hkv, d=d, bs=bs, int8=int8,
                split_tokens=split, max_blocks=max_blocks, num_blocks=max(blocks, 1), fused_step=fused,
                graph=graph), steps


@pytest.mark.parametrize("i", range(24))
def test_random_shape_matches_oracle(i):
    kw, steps = _case(i)
    w = Workload(**kw)
    for t in range(steps):
        out = w.step().float().cpu().numpy()
        for b in range(w.B):
            assert_close(out[0, b], w.oracle_out(0, b, t), f"case {i} {kw} step {t} seq {b}")
    assert w.error_bits() == 0
    for b in range(w.B):
        w.check_pool_bytes(0, b, w.prior[b] + steps)
