"""The trace driver's batch order (host logic, no GPU)."""

import os
import sys
from types import SimpleNamespace

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from paged_kv_cache_56_gb300.trace import TraceDriver  # noqa: E402


def _order(lengths):
    running = [SimpleNamespace(rid=100 + i, length=n) for i, n in enumerate(lengths)]
    rids = TraceDriver.batch_order(SimpleNamespace(running=running))
    return [lengths[r - 100] for r in rids]


def test_shortest_quarter_first_then_longest_first():
    assert _order([5, 9, 1, 7, 3, 8, 2, 6]) == [1, 2, 9, 8, 7, 6, 5, 3]


def test_every_request_once():
    lengths = list(range(37, 0, -3)) + [4, 4, 4]
    got = _order(lengths)
    assert sorted(got) == sorted(lengths)
    k = len(lengths) // 4
    assert got[:k] == sorted(lengths)[:k]
    assert got[k:] == sorted(lengths)[k:][::-1]


def test_small_batches():
    assert _order([]) == []
    assert _order([7]) == [7]
    assert _order([3, 9, 5]) == [9, 5, 3]  # fewer than four: longest first
