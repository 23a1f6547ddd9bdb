"""Pins of the oracle's contiguous histories: when blocks quantize, what the
context holds, and that chunked and token-by-token appends agree."""

import numpy as np
import torch

from oracle.cache import SequenceHistory
from oracle.quantize import quantize_block


def _rows(gen, n, hkv, d):
    return (torch.randn(n, hkv, d, generator=gen) * 2).to(torch.bfloat16).float().numpy()


def test_blocks_quantize_exactly_when_they_fill():
    gen = torch.Generator().manual_seed(0)
    h = SequenceHistory(2, 8, 16, int8=True)
    k, v = _rows(gen, 40, 2, 8), _rows(gen, 40, 2, 8)
    for t in range(40):
        filled = h.append(k[t:t + 1], v[t:t + 1])
        assert filled == ([t // 16] if (t + 1) % 16 == 0 else [])
        assert sorted(h.blocks) == list(range((t + 1) // 16))
    # block i's codes are the quantizer applied to rows i*16..i*16+15 of each head
    for i in range(2):
        qk, sk, qv, sv = h.blocks[i]
        for g in range(2):
            q_ref, s_ref = quantize_block(k[i * 16:(i + 1) * 16, g])
            assert np.array_equal(qk[g], q_ref) and sk[g] == s_ref
            q_ref, s_ref = quantize_block(v[i * 16:(i + 1) * 16, g])
            assert np.array_equal(qv[g], q_ref) and sv[g] == s_ref


def test_context_dequantizes_full_blocks_and_keeps_tail():
    gen = torch.Generator().manual_seed(1)
    h = SequenceHistory(2, 8, 16, int8=True)
    k, v = _rows(gen, 37, 2, 8), _rows(gen, 37, 2, 8)
    h.append(k, v)
    kh, vh = h.context()
    assert kh.shape == (37, 2, 8)
    assert np.array_equal(kh[32:], k[32:].astype(np.float64))
    assert np.array_equal(vh[32:], v[32:].astype(np.float64))
    qk, sk, _, _ = h.blocks[1]
    assert np.array_equal(kh[16:32, 1], qk[1].astype(np.float64) * np.float64(sk[1]))
    assert not np.array_equal(kh[:32], k[:32])  # quantization changed something
    assert np.abs(kh[:32] - k[:32]).max() <= np.max([h.blocks[i][1].max() for i in range(2)])


def test_bf16_mode_context_is_raw():
    gen = torch.Generator().manual_seed(2)
    h = SequenceHistory(1, 4, 16, int8=False)
    k, v = _rows(gen, 33, 1, 4), _rows(gen, 33, 1, 4)
    assert h.append(k, v) == [0, 1]
    assert h.blocks == {}
    kh, vh = h.context()
    assert np.array_equal(kh, k.astype(np.float64)) and np.array_equal(vh, v.astype(np.float64))


def test_chunked_equals_token_by_token():
    gen = torch.Generator().manual_seed(3)
    k, v = _rows(gen, 150, 2, 8), _rows(gen, 150, 2, 8)
    a = SequenceHistory(2, 8, 64, int8=True)
    a.append(k, v)
    b = SequenceHistory(2, 8, 64, int8=True)
    for s in range(0, 150, 7):
        b.append(k[s:s + 7], v[s:s + 7])
    assert sorted(a.blocks) == sorted(b.blocks) == [0, 1]
    for i in a.blocks:
        for x, y in zip(a.blocks[i], b.blocks[i]):
            assert np.array_equal(x, y)
    assert all(np.array_equal(x, y) for x, y in zip(a.context(), b.context()))
