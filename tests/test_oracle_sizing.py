"""Pins of the oracle's closed-form sizing against the numbers the pages print."""

import os

import pytest

from oracle import sizing

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sizing_pins.txt")
GIB = 2 ** 30


def _cases():
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split("=")
            name, *args = lhs.split()
            yield name, args, int(rhs)


@pytest.mark.parametrize("name,args,expected", list(_cases()))
def test_golden_sizing(name, args, expected):
    if name == "kv_bytes":
        got = sizing.kv_bytes(*map(int, args))
    elif name == "kv_bytes_per_token":
        got = sizing.kv_bytes_per_token(*map(int, args))
    elif name == "max_concurrent_requests_gib":
        mem, util, weights, per_tok, max_len = args
        got = sizing.max_concurrent_requests(float(mem) * GIB, float(util), float(weights) * GIB,
                                             int(per_tok), int(max_len))
    elif name == "blocks_needed":
        got = sizing.blocks_needed(*map(int, args))
    elif name == "paged_tail_waste":
        got = sizing.paged_tail_waste(*map(int, args))
    elif name == "fixed_bucket_waste_permille":
        got = int(sizing.fixed_bucket_waste_fraction(int(args[0])) * 1000)
    else:
        raise AssertionError(name)
    assert got == expected


def test_printed_roundings():
    # The pages print truncated decimal gigabytes: 3.6GB, 1.8GB; 512KB and 50GB are binary.
    assert f"{sizing.kv_bytes(28, 8, 128, 8000, 4, 2) / 1e9:.3f}".startswith("3.6")
    assert f"{sizing.kv_bytes(28, 8, 128, 8000, 4, 1) / 1e9:.3f}".startswith("1.8")
    assert sizing.kv_bytes_per_token(32, 32, 128, 2) == 512 * 1024
    assert sizing.kv_bytes(32, 32, 128, 1024, 100, 2) == 50 * GIB
    # 2 GB per 4096-token request at 512KB/token
    assert sizing.kv_bytes_per_token(32, 32, 128, 2) * 4096 == 2 * GIB
    # 80 GB * 0.9 - 14 GB = 58 GB
    assert 80 * GIB * 0.9 - 14 * GIB == 58 * GIB


def test_int8_halves_every_size():
    for args in [(28, 8, 128, 8000, 4), (32, 32, 128, 1024, 100), (1, 1, 64, 17, 3)]:
        assert sizing.kv_bytes(*args, 1) * 2 == sizing.kv_bytes(*args, 2)


def test_tail_waste_bound_all_lengths():
    for bs in (16, 64):
        for n in range(1, 5000):
            w = sizing.paged_tail_waste(n, bs)
            assert 0 <= w < bs
            assert (n + w) % bs == 0
            assert sizing.blocks_needed(n, bs) * bs >= n > (sizing.blocks_needed(n, bs) - 1) * bs


def test_blocks_needed_edges():
    assert sizing.blocks_needed(0, 16) == 0
    assert sizing.blocks_needed(1, 16) == 1
    assert sizing.blocks_needed(16, 16) == 1
    assert sizing.blocks_needed(17, 16) == 2
    with pytest.raises(ValueError):
        sizing.blocks_needed(5, 0)
