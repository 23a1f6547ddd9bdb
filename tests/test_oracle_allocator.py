"""Pins of the oracle allocator: a hand-worked trace and invariants."""

import os
import random

import pytest

from oracle.allocator import (FreeBlockPool, OutOfBlocks, UnknownRequest, DuplicateRequest)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "allocator_trace.txt")
COW_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "cow_trace.txt")


def _run_golden(path=GOLDEN):
    pool = None
    with open(path) as f:
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


def test_cow_golden_trace():
    n = 0
    for pool, op, args, want in _run_golden(COW_GOLDEN):
        n += 1
        try:
            if op == "alloc":
                got = [str(b) for b in pool.alloc(args[0], int(args[1]))]
            elif op == "append":
                b = pool.append_block(args[0])
                got = ["EMPTY"] if b is None else [str(b)]
            elif op == "free":
                got = [str(b) for b in pool.free(args[0])]
            elif op == "fork":
                pool.fork(args[0], args[1])
                got = []
            elif op == "cow":
                r = pool.cow(args[0], int(args[1]))
                got = ["NONE"] if r is None else [str(r[0]), str(r[1])]
            elif op == "refs":
                got = [str(pool.refs(int(args[0])))]
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
        assert got == want, (op, args, got)
    assert n > 20


def test_random_forks_keep_reference_counts():
    """Random alloc / append / fork / cow / free: every block is free xor held,
    a block's count is the number of requests holding it, a cow leaves the
    writer's block held by it alone, and freeing everything restores the pool."""
    rng = random.Random(11)
    pool = FreeBlockPool(40, initial_order=rng.sample(range(40), 40))
    live, nxt = [], 0
    for _ in range(3000):
        op = rng.random()
        try:
            if op < 0.2 or not live:
                pool.alloc(nxt, rng.randint(0, 4))
                live.append(nxt)
                nxt += 1
            elif op < 0.4:
                pool.append_block(rng.choice(live))
            elif op < 0.55:
                pool.fork(rng.choice(live), nxt)
                live.append(nxt)
                nxt += 1
            elif op < 0.8:
                r = rng.choice(live)
                t = pool.table(r)
                if t:
                    i = rng.randrange(len(t))
                    before = pool.refs(t[i])
                    res = pool.cow(r, i)
                    t2 = pool.table(r)
                    assert (res is None) == (before == 1)
                    assert pool.refs(t2[i]) == 1
                    if res is not None:
                        assert res == (t[i], t2[i]) and pool.refs(t[i]) == before - 1
            else:
                r = rng.choice(live)
                held = set(pool.table(r))
                back = pool.free(r)
                live.remove(r)
                assert set(back) == {b for b in held if pool.refs(b) == 0}
        except OutOfBlocks:
            pass
        held = {b for r in pool.private for b in pool.private[r]}
        assert held.isdisjoint(pool.free_list)
        assert sorted(held | set(pool.free_list)) == list(range(40))
        assert len(pool.free_list) == len(set(pool.free_list))
    for r in list(live):
        pool.free(r)
    assert sorted(pool.free_list) == list(range(40))


def test_cow_of_attached_prefix_is_rejected():
    pool = FreeBlockPool(8)
    pool.alloc("prefix", 2)
    pool.alloc("A", 1)
    pool.attach_shared("A", [0, 1])
    with pytest.raises(ValueError):
        pool.cow("A", 1)
    assert pool.cow("A", 2) is None
