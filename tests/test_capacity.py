"""The capacity study (host arithmetic) against the oracle's closed forms and
the pages' sizing figures: 512 KB per token and 29 requests at 58 GB for
max-length reservation ("vLLM核心概念" §3.1, §3.5), more than 40% padding for
600 tokens in a 1024 bucket and less than one block of waste when paged
("无 vLLM 环境下的 Paged-KV" §1.1-1.2)."""

import pytest

from oracle import sizing
from paged_kv_cache_56_gb300.capacity import (BUCKETS, KVShape, concurrency, reserved_bytes, study,
                                              trace_lengths)

SEVEN_B = KVShape(layers=32, kv_heads=32, head_dim=128)
GIB = 2 ** 30


def test_per_token_bytes_match_the_formula():
    assert SEVEN_B.bytes_per_token(2) == sizing.kv_bytes_per_token(32, 32, 128, 2) == 524288
    assert SEVEN_B.bytes_per_token(1) * 2 == SEVEN_B.bytes_per_token(2)


def test_max_len_reservation_gives_the_pages_29():
    budget = int(80 * 0.9 * GIB - 14 * GIB)
    want = sizing.max_concurrent_requests(80 * GIB, 0.9, 14 * GIB, 524288, 4096)
    assert want == 29
    assert concurrency([1] * 100, budget, "max_len", SEVEN_B, max_len=4096) == want
    assert concurrency(trace_lengths(3, 100), budget, "max_len", SEVEN_B) == want


def test_bucket_and_paged_waste():
    tok = SEVEN_B.bytes_per_token(2)
    assert reserved_bytes(600, "bucket", SEVEN_B, buckets=(128, 256, 512, 1024)) == 1024 * tok
    assert sizing.fixed_bucket_waste_fraction(600) > 0.40
    for ell in range(0, 5000, 7):
        got = reserved_bytes(ell, "paged", SEVEN_B, block_size=16) // tok - ell
        assert got == sizing.paged_tail_waste(ell, 16) < 16
    assert reserved_bytes(600, "paged", SEVEN_B) == sizing.blocks_needed(600, 16) * 16 * tok == 38 * 16 * tok


def test_int8_blocks_hold_scales_and_a_bf16_tail():
    s = KVShape(layers=28, kv_heads=8, head_dim=128)
    got = reserved_bytes(8001, "paged_int8", s, block_size=16)
    full = 8001 // 16
    want = full * 16 * s.bytes_per_token(1) + full * 28 * 8 * 2 * 4 + 16 * s.bytes_per_token(2)
    assert got == want
    with pytest.raises(ValueError):
        reserved_bytes(5000, "bucket", s, buckets=BUCKETS)


def test_schemes_rank_as_the_pages_say():
    lengths = trace_lengths(1234, 4000)
    r = study(lengths, 58 * GIB, SEVEN_B)
    n = {k: v["requests"] for k, v in r.items()}
    assert n["max_len"] == 29
    assert n["max_len"] < n["bucket"] < n["paged"] < n["paged_int8"]
    assert 1.8 < n["paged_int8"] / n["paged"] <= 2.1
    assert r["paged"]["waste"] < 0.02 < r["bucket"]["waste"]
