"""Pins of the oracle allocator: a hand-worked trace and invariants."""

import os
import random

import pytest

from oracle.allocator import (FreeBlockPool, OutOfBlocks, UnknownRequest, DuplicateRequest)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "allocator_trace.txt")


def _run_golden():
    pool = None
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#")[0].rstrip()
            if not line.strip():
                continue
            if line.startswith("pool"):
                pool = FreeBlockPool(int(line.split()[1]))
                continue
            lhs, rhs = line.split("->")
            rhs = rhs.split()
            op, *args = lhs.split()
            yield pool, op, args, rhs


def test_golden_trace():
    n = 0
    for pool, op, args, want in _run_golden():
        n += 1
        try:
            if op == "alloc":
                got = [str(b) for b in pool.alloc(args[0], int(args[1]))]
            elif op == "append":
                b = pool.append_block(args[0])
                got = ["EMPTY"] if b is None else [str(b)]
            elif op == "free":
                got = [str(b) for b in pool.free(args[0])]
            elif op == "free_list":
                got = [str(b) for b in pool.free_list]
            elif op == "table":
                got = [str(b) for b in pool.table(args[0])]
            else:
                raise AssertionError(op)
        except OutOfBlocks:
            got = ["OOM"]
        except DuplicateRequest:
            got = ["DUP"]
        except UnknownRequest:
            got = ["UNKNOWN"]
        assert got == want, (op, args)
    assert n > 15


def _check_conservation(pool):
    held = [b for r in pool.private for b in pool.private[r]]
    everything = sorted(held + pool.free_list)
    assert everything == list(range(pool.total_blocks))


def test_random_ops_conserve_blocks_and_fifo():
    rng = random.Random(5)
    pool = FreeBlockPool(64, initial_order=rng.sample(range(64), 64))
    live = []
    for i in range(20000):
        op = rng.random()
        if op < 0.3:
            n = rng.randint(0, 12)
            before = list(pool.free_list)
            try:
                got = pool.alloc(i, n)
                assert got == before[:n]
                live.append(i)
            except OutOfBlocks:
                assert len(before) < n and pool.free_list == before
        elif op < 0.7 and live:
            r = rng.choice(live)
            before = list(pool.free_list)
            b = pool.append_block(r)
            if before:
                assert b == before[0] and pool.private[r][-1] == b
            else:
                assert b is None
        elif live:
            r = live.pop(rng.randrange(len(live)))
            before = list(pool.free_list)
            held = list(pool.private[r])
            assert pool.free(r) == held
            assert pool.free_list == before + held
        _check_conservation(pool)


def test_errors_leave_state_unchanged():
    pool = FreeBlockPool(4)
    pool.alloc(1, 2)
    snap = (list(pool.free_list), {k: list(v) for k, v in pool.private.items()})
    with pytest.raises(OutOfBlocks):
        pool.alloc(2, 3)
    with pytest.raises(DuplicateRequest):
        pool.alloc(1, 1)
    with pytest.raises(UnknownRequest):
        pool.free(9)
    with pytest.raises(UnknownRequest):
        pool.append_block(9)
    assert (pool.free_list, pool.private) == snap


def test_shared_prefix_blocks_are_not_freed():
    pool = FreeBlockPool(10)
    prefix = pool.alloc("prefix", 3)
    pool.alloc("r1", 2)
    pool.attach_shared("r1", prefix)
    pool.alloc("r2", 1)
    pool.attach_shared("r2", prefix)
    assert pool.table("r1") == prefix + [3, 4]
    assert pool.table("r2") == prefix + [5]
    assert pool.free("r1") == [3, 4]
    assert pool.free_list == [6, 7, 8, 9, 3, 4]
    assert pool.table("r2") == prefix + [5]
    rows = pool.block_tables(["r2", "prefix"], 6)
    assert rows == [[0, 1, 2, 5, -1, -1], [0, 1, 2, -1, -1, -1]]
    with pytest.raises(ValueError):
        pool.block_tables(["r2"], 3)


def test_page_example_600_tokens():
    # 600 tokens in 16-token blocks take 38 blocks; the tail block wastes 8 slots.
    pool = FreeBlockPool(2048)
    ids = pool.alloc("s", 38)
    assert len(ids) == 38 and pool.num_free() == 2048 - 38
    assert 38 * 16 - 600 == 8 < 16
