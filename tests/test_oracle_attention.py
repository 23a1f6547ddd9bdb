"""Pins of the oracle's decode attention: a pure-Python brute force, closed
forms and invariants, and the identity that merging the softmax states of a
partition reproduces the whole."""

import math
import random

import numpy as np
import pytest

from oracle.attention import decode_attention, partial_state, merge_partials, kv_head_of


def _brute(q, k, v, sm_scale):
    """Scalar loops with math.exp/math.fsum: independent of the numpy path."""
    hq, d = len(q), len(q[0])
    n, hkv = len(k), len(k[0])
    g = hq // hkv
    out = []
    for h in range(hq):
        kh = h // g
        s = [math.fsum(q[h][i] * k[t][kh][i] for i in range(d)) * sm_scale for t in range(n)]
        mx = max(s)
        e = [math.exp(x - mx) for x in s]
        z = math.fsum(e)
        out.append([math.fsum(e[t] / z * v[t][kh][i] for t in range(n)) for i in range(d)])
    return np.array(out)


@pytest.mark.parametrize("hq,hkv,d,n", [(4, 2, 8, 1), (4, 2, 8, 2), (4, 2, 8, 15), (4, 2, 8, 17),
                                        (4, 4, 4, 9), (8, 1, 4, 20), (6, 3, 5, 7)])
def test_brute_force_tiny(hq, hkv, d, n):
    rng = random.Random(hq * 1000 + n)
    q = [[rng.gauss(0, 1) for _ in range(d)] for _ in range(hq)]
    k = [[[rng.gauss(0, 2) for _ in range(d)] for _ in range(hkv)] for _ in range(n)]
    v = [[[rng.gauss(0, 1) for _ in range(d)] for _ in range(hkv)] for _ in range(n)]
    sm = 1 / math.sqrt(d)
    got = decode_attention(np.array(q), np.array(k), np.array(v), sm)
    assert np.allclose(got, _brute(q, k, v, sm), rtol=1e-12, atol=1e-12)


def test_two_token_closed_form():
    # q = e0, k0 = a e0, k1 = b e0: w1 = 1 / (1 + exp((a - b) * sm_scale)).
    d, a, b, sm = 4, 1.5, -0.5, 0.3
    q = np.zeros((1, d)); q[0, 0] = 1.0
    k = np.zeros((2, 1, d)); k[0, 0, 0] = a; k[1, 0, 0] = b
    v = np.zeros((2, 1, d)); v[0, 0] = [1, 0, 0, 0]; v[1, 0] = [0, 1, 0, 0]
    out, w = decode_attention(q, k, v, sm, return_weights=True)
    w1 = 1 / (1 + math.exp((a - b) * sm))
    assert math.isclose(w[0, 1], w1, rel_tol=1e-14)
    assert np.allclose(out[0], [1 - w1, w1, 0, 0], atol=1e-15)


def test_single_token_returns_its_value():
    rng = np.random.default_rng(0)
    q = rng.normal(size=(8, 16)); k = rng.normal(size=(1, 2, 16)); v = rng.normal(size=(1, 2, 16))
    out = decode_attention(q, k, v, 0.25)
    for h in range(8):
        assert np.array_equal(out[h], v[0, h // 4])


def test_constant_values_and_zero_keys():
    rng = np.random.default_rng(1)
    n, hkv, d = 37, 2, 8
    q = rng.normal(size=(4, d)) * 3
    k = rng.normal(size=(n, hkv, d)) * 3
    c = rng.normal(size=(hkv, d))
    v = np.broadcast_to(c, (n, hkv, d)).copy()
    out = decode_attention(q, k, v, 0.5)
    for h in range(4):
        assert np.allclose(out[h], c[h // 2], atol=1e-12)
    v = rng.normal(size=(n, hkv, d))
    out = decode_attention(q, np.zeros_like(k), v, 0.5)
    for h in range(4):
        assert np.allclose(out[h], v[:, h // 2].mean(axis=0), atol=1e-12)


def test_gqa_grouping_is_contiguous():
    n, d = 5, 4
    k = np.random.default_rng(2).normal(size=(n, 2, d))
    v = np.zeros((n, 2, d)); v[:, 0] = 1.0; v[:, 1] = 2.0
    out = decode_attention(np.ones((4, d)), k, v, 1.0)
    assert np.allclose(out[:, 0], [1, 1, 2, 2])
    assert [kv_head_of(h, 4, 2) for h in range(4)] == [0, 0, 1, 1]
    with pytest.raises(ValueError):
        kv_head_of(0, 6, 4)


def test_weights_sum_to_one_and_permutation_invariance():
    rng = np.random.default_rng(3)
    n, hkv, d = 200, 2, 16
    q = rng.normal(size=(4, d)) * 4
    k = rng.normal(size=(n, hkv, d)) * 4
    v = rng.normal(size=(n, hkv, d))
    out, w = decode_attention(q, k, v, 1 / 4, return_weights=True)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-14)
    assert (w >= 0).all()
    perm = rng.permutation(n)
    out2 = decode_attention(q, k[perm], v[perm], 1 / 4)
    assert np.allclose(out, out2, atol=1e-13)


@pytest.mark.parametrize("base", [math.e, 2.0])
def test_merge_of_partition_equals_whole(base):
    rng = np.random.default_rng(4)
    n, d = 301, 8
    q = rng.normal(size=d) * 3
    k = rng.normal(size=(n, d)) * 3
    v = rng.normal(size=(n, d))
    whole = decode_attention(q[None], k[:, None], v[:, None], 0.35)[0]
    for parts in (1, 2, 7, 301):
        cuts = sorted(rng.choice(np.arange(1, n), size=parts - 1, replace=False)) if parts > 1 else []
        bounds = [0, *cuts, n]
        states = [partial_state(q, k[a:b], v[a:b], 0.35, base=base) for a, b in zip(bounds, bounds[1:])]
        ms, ls, os_ = zip(*states)
        assert np.allclose(merge_partials(ms, ls, os_, base=base), whole, atol=1e-13)


def test_empty_context_rejected():
    with pytest.raises(ValueError):
        decode_attention(np.ones((2, 4)), np.ones((0, 1, 4)), np.ones((0, 1, 4)), 1.0)
