"""The C ABI on the host: exported symbols, argument validation that returns
before any CUDA call, and the C++ allocator against the oracle allocator."""

import ctypes
import os
import random
import re

import numpy as np
import pytest

from libpkv import ensure_built
from oracle.allocator import FreeBlockPool, OutOfBlocks, UnknownRequest, DuplicateRequest
from paged_kv_cache_56_gb300 import pkv

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "pkv.h")


@pytest.fixture(scope="module")
def L():
    return ensure_built()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = _declared_functions()
    assert len(names) >= 17
    for n in names:
        assert hasattr(L, n), n
    assert sorted(pkv.EXPORTED) == names


def test_desc_layout_matches_header():
    # 5 pointers, 7 int32, 1 pointer (with padding before it)
    assert ctypes.sizeof(pkv.CacheDesc) == 5 * 8 + 7 * 4 + 4 + 8


def _desc(**kw):
    d = dict(k_pool=16, v_pool=32, scales=None, k_tail=None, v_tail=None, num_blocks=4, num_q_heads=4,
             num_kv_heads=2, head_dim=128, block_size=16, max_slots=0, dtype=pkv.PKV_DTYPE_BF16, err_word=None)
    d.update(kw)
    return pkv.CacheDesc(**d)


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=96), pkv.PKV_ERR_UNSUPPORTED),
    (dict(block_size=32), pkv.PKV_ERR_UNSUPPORTED),
    (dict(num_q_heads=6, num_kv_heads=4), pkv.PKV_ERR_UNSUPPORTED),
    (dict(num_q_heads=32, num_kv_heads=2), pkv.PKV_ERR_UNSUPPORTED),   # G = 16
    (dict(k_pool=None), pkv.PKV_ERR_INVALID),
    (dict(k_pool=24), pkv.PKV_ERR_INVALID),                           # misaligned pool
    (dict(dtype=7), pkv.PKV_ERR_INVALID),
    (dict(dtype=pkv.PKV_DTYPE_INT8), pkv.PKV_ERR_INVALID),            # INT8 without tails/scales
])
def test_descriptor_validation(L, kw, code):
    d = _desc(**kw)
    rc = L.pkv_decode_attention(ctypes.byref(d), 16, 16, 4, 16, 16, 1, 0.1, 0, 0, None, None, None, 16, None)
    assert rc == code
    rc = L.pkv_append_kv(ctypes.byref(d), 16, 16, 16, 16, 16, 1, None)
    assert rc == code


def test_argument_validation(L):
    d = _desc()
    attn = L.pkv_decode_attention
    assert attn(None, 16, 16, 4, 16, 16, 1, 0.1, 0, 0, None, None, None, 16, None) == pkv.PKV_ERR_INVALID
    assert attn(ctypes.byref(d), 16, 16, 4, 16, 16, 0, 0.1, 0, 0, None, None, None, 16, None) == pkv.PKV_OK  # B = 0
    assert attn(ctypes.byref(d), None, 16, 4, 16, 16, 1, 0.1, 0, 0, None, None, None, 16, None) == pkv.PKV_ERR_INVALID
    assert attn(ctypes.byref(d), 16, 16, 0, 16, 16, 1, 0.1, 0, 0, None, None, None, 16, None) == pkv.PKV_ERR_INVALID
    assert attn(ctypes.byref(d), 16, 16, 4, 16, 16, 1, float("nan"), 0, 0, None, None, None, 16, None) == pkv.PKV_ERR_INVALID
    # split must be a multiple of block size and of 16; max_splits must cover max_blocks * bs
    assert attn(ctypes.byref(d), 16, 16, 4, 16, 16, 1, 0.1, 24, 8, 16, 16, None, 16, None) == pkv.PKV_ERR_INVALID
    assert attn(ctypes.byref(d), 16, 16, 4, 16, 16, 1, 0.1, 32, 1, 16, 16, None, 16, None) == pkv.PKV_ERR_INVALID
    assert attn(ctypes.byref(d), 16, 16, 4, 16, 16, 1, 0.1, 32, 2, None, 16, None, 16, None) == pkv.PKV_ERR_INVALID
    # misaligned split-K arrival counters
    assert attn(ctypes.byref(d), 16, 16, 4, 16, 16, 1, 0.1, 32, 2, 16, 16, 18, 16, None) == pkv.PKV_ERR_INVALID
    assert L.pkv_decode_ctas_per_sm(ctypes.byref(_desc(head_dim=80)), 0, 4) == pkv.PKV_ERR_UNSUPPORTED
    assert L.pkv_decode_ctas_per_sm(ctypes.byref(d), 24, 4) == pkv.PKV_ERR_INVALID
    assert L.pkv_append_kv(ctypes.byref(d), 16, 16, 16, 16, 16, 0, None) == pkv.PKV_OK  # T = 0
    assert L.pkv_append_kv(ctypes.byref(d), 16, 16, None, 16, 16, 3, None) == pkv.PKV_ERR_INVALID
    assert L.pkv_quantize_full_blocks(ctypes.byref(d), 16, 16, 1, None) == pkv.PKV_ERR_INVALID  # BF16 cache
    assert L.pkv_copy_blocks(ctypes.byref(d), 16, 16, 0, None) == pkv.PKV_OK  # n = 0
    assert L.pkv_copy_blocks(ctypes.byref(d), 16, 16, -1, None) == pkv.PKV_ERR_INVALID
    assert L.pkv_copy_blocks(ctypes.byref(d), None, 16, 2, None) == pkv.PKV_ERR_INVALID
    assert L.pkv_copy_blocks(None, 16, 16, 2, None) == pkv.PKV_ERR_INVALID
    assert L.pkv_copy_slots(ctypes.byref(d), 16, 16, 2, None) == pkv.PKV_ERR_INVALID  # BF16 cache: no tails
    assert L.pkv_splitk_reduce(16, 16, 16, 1, 4, 96, 16, 2, 16, None) == pkv.PKV_ERR_UNSUPPORTED
    assert L.pkv_splitk_reduce(16, 16, 16, 1, 4, 128, 0, 2, 16, None) == pkv.PKV_ERR_INVALID
    assert pkv.pkv_splitk_ws_o_bytes(2, 3, 128, 5) == 2 * 3 * 5 * 128 * 4
    assert pkv.pkv_splitk_ws_ml_bytes(2, 3, 5) == 2 * 3 * 5 * 2 * 4
    # the no-allocation entry point rejects a negative split like the regular one
    static = L.pkv_decode_attention_static_ws
    assert static(ctypes.byref(d), 16, 16, 4, 16, 16, 1, 0.1, -16, 2, 16, None) == pkv.PKV_ERR_INVALID
    assert attn(ctypes.byref(d), 16, 16, 4, 16, 16, 1, 0.1, -16, 2, 16, 16, None, 16, None) == pkv.PKV_ERR_INVALID
    # appended rows are read 16 bytes at a time: a misaligned k_new / v_new is refused
    layers = L.pkv_decode_layers
    assert layers(ctypes.byref(d), 1, 16, 0, 24, 32, 0, 16, 0, 16, 4, 16, 16, 1, 0.1, 0, 0,
                  None, None, None, None) == pkv.PKV_ERR_INVALID
    assert layers(ctypes.byref(d), 1, 16, 0, 32, 40, 0, 16, 0, 16, 4, 16, 16, 1, 0.1, 0, 0,
                  None, None, None, None) == pkv.PKV_ERR_INVALID
    assert L.pkv_decode_step(ctypes.byref(d), 16, 24, 32, 16, 4, 16, 16, 1, 0.1, 0, 0, None, None, None,
                             16, None) == pkv.PKV_ERR_INVALID
    # the error-word reader: bad counts and a NULL array are refused before any CUDA call
    bits = ctypes.c_int32(7)
    assert L.pkv_sync_status(None, 1, None, ctypes.byref(bits)) == pkv.PKV_ERR_INVALID
    assert L.pkv_sync_status(ctypes.byref(d), -1, None, ctypes.byref(bits)) == pkv.PKV_ERR_INVALID
    assert bits.value == 0


def test_status_codes_match_header():
    """The binding's status constants are the header's, and the device-timeout
    status has the value the boundary fixes for it (-7), distinct from every
    other status."""
    src = open(HEADER).read()
    codes = {m.group(1): int(m.group(2)) for m in re.finditer(r"#define\s+(PKV_(?:OK|ERR_\w+))\s+(-?\d+)", src)}
    assert codes["PKV_OK"] == 0 and codes["PKV_ERR_DEVICE_TIMEOUT"] == -7
    assert len(set(codes.values())) == len(codes)
    for name, value in codes.items():
        assert getattr(pkv, name) == value, name
    bits = {m.group(1): int(m.group(2)) for m in re.finditer(r"#define\s+(PKV_DEVERR_\w+)\s+(\d+)", src)}
    for name, value in bits.items():
        assert getattr(pkv, name) == value, name


def test_binding_refuses_host_tensors():
    import torch
    d = _desc()
    with pytest.raises(ValueError):
        pkv.pkv_decode_attention(d, torch.zeros(4, 128, dtype=torch.bfloat16), torch.zeros(1, 4, dtype=torch.int32),
                                 torch.ones(1, dtype=torch.int32), None, 0.1,
                                 torch.zeros(4, 128, dtype=torch.bfloat16))


# -- allocator -----------------------------------------------------------------

def test_allocator_replays_oracle_ids(L):
    rng = random.Random(1234)
    n = 97
    order = rng.sample(range(n), n)
    h = pkv.pkv_allocator_create(n, 16, order)
    ref = FreeBlockPool(n, order)
    live = []
    try:
        for i in range(100_000):
            u = rng.random()
            if u < 0.3:
                k = rng.randint(0, 9)
                try:
                    want = ref.alloc(i, k)
                except OutOfBlocks:
                    with pytest.raises(pkv.PkvError) as e:
                        pkv.pkv_alloc(h, i, k)
                    assert e.value.code == pkv.PKV_ERR_OOM
                else:
                    assert pkv.pkv_alloc(h, i, k) == want
                    live.append(i)
            elif u < 0.75 and live:
                r = rng.choice(live)
                want = ref.append_block(r)
                if want is None:
                    with pytest.raises(pkv.PkvError) as e:
                        pkv.pkv_append_block(h, r)
                    assert e.value.code == pkv.PKV_ERR_OOM
                else:
                    assert pkv.pkv_append_block(h, r) == want
            elif live:
                r = live.pop(rng.randrange(len(live)))
                ref.free(r)
                pkv.pkv_free(h, r)
            if i % 997 == 0:
                assert pkv.pkv_free_list(h) == ref.free_list
                for r in live[:5]:
                    assert pkv.pkv_request_table(h, r) == ref.table(r)
        assert pkv.pkv_num_free(h) == ref.num_free()
        assert pkv.pkv_free_list(h) == ref.free_list
    finally:
        pkv.pkv_allocator_destroy(h)


def test_allocator_errors_and_shared_blocks(L):
    h = pkv.pkv_allocator_create(10, 16)
    ref = FreeBlockPool(10)
    try:
        prefix = pkv.pkv_alloc(h, -1, 3)
        assert prefix == ref.alloc(-1, 3)
        for r in (5, 6):
            assert pkv.pkv_alloc(h, r, 1) == ref.alloc(r, 1)
            pkv.pkv_attach_shared(h, r, prefix)
            ref.attach_shared(r, prefix)
        assert pkv.pkv_request_table(h, 5) == ref.table(5) == prefix + [3]
        for fn, args, code in [(pkv.pkv_alloc, (5, 1), pkv.PKV_ERR_EXISTS),
                               (pkv.pkv_free, (77,), pkv.PKV_ERR_NOT_FOUND),
                               (pkv.pkv_append_block, (77,), pkv.PKV_ERR_NOT_FOUND),
                               (pkv.pkv_alloc, (8, 6), pkv.PKV_ERR_OOM),
                               (pkv.pkv_attach_shared, (5, [10]), pkv.PKV_ERR_INVALID)]:
            with pytest.raises(pkv.PkvError) as e:
                fn(h, *args)
            assert e.value.code == code
        assert pkv.pkv_free_list(h) == ref.free_list
        pkv.pkv_free(h, 5)
        ref.free(5)
        assert pkv.pkv_free_list(h) == ref.free_list == [5, 6, 7, 8, 9, 3]
        tab = pkv.pkv_build_block_tables(h, [6, -1], 5)
        assert tab.tolist() == [prefix + [4, -1], prefix + [-1, -1]]
        with pytest.raises(pkv.PkvError) as e:
            pkv.pkv_build_block_tables(h, [6], 3)
        assert e.value.code == pkv.PKV_ERR_INVALID
        with pytest.raises(pkv.PkvError) as e:
            pkv.pkv_build_block_tables(h, [5], 8)
        assert e.value.code == pkv.PKV_ERR_NOT_FOUND
    finally:
        pkv.pkv_allocator_destroy(h)


def test_allocator_create_rejects_bad_order(L):
    with pytest.raises(pkv.PkvError):
        pkv.pkv_allocator_create(4, 16, [0, 1, 1, 2])
    with pytest.raises(pkv.PkvError):
        pkv.pkv_allocator_create(0, 16)


def test_page_sizing_through_the_allocator(L):
    # A 600-token sequence in 16-token blocks holds 38 blocks (tail waste 8 < 16).
    h = pkv.pkv_allocator_create(2048, 16)
    try:
        ids = pkv.pkv_alloc(h, 1, -(-600 // 16))
        assert len(ids) == 38 and pkv.pkv_num_free(h) == 2010
    finally:
        pkv.pkv_allocator_destroy(h)


def test_forks_and_cow_replay_oracle_ids(L):
    """Random alloc / append / fork / cow / free through the C ABI and through
    the oracle pool: identical ids, tables, free lists and reference counts."""
    rng = random.Random(99)
    n = 61
    order = rng.sample(range(n), n)
    h = pkv.pkv_allocator_create(n, 16, order)
    ref = FreeBlockPool(n, order)
    live, nxt = [], 0
    try:
        for i in range(20_000):
            u = rng.random()
            if u < 0.15 or not live:
                k = rng.randint(0, 5)
                try:
                    want = ref.alloc(nxt, k)
                except OutOfBlocks:
                    with pytest.raises(pkv.PkvError) as e:
                        pkv.pkv_alloc(h, nxt, k)
                    assert e.value.code == pkv.PKV_ERR_OOM
                else:
                    assert pkv.pkv_alloc(h, nxt, k) == want
                    live.append(nxt)
                nxt += 1
            elif u < 0.35:
                r = rng.choice(live)
                want = ref.append_block(r)
                if want is None:
                    with pytest.raises(pkv.PkvError):
                        pkv.pkv_append_block(h, r)
                else:
                    assert pkv.pkv_append_block(h, r) == want
            elif u < 0.5:
                r = rng.choice(live)
                ref.fork(r, nxt)
                pkv.pkv_fork(h, r, nxt)
                live.append(nxt)
                nxt += 1
            elif u < 0.8:
                r = rng.choice(live)
                t = ref.table(r)
                if t:
                    idx = rng.randrange(len(t))
                    try:
                        want = ref.cow(r, idx)
                    except OutOfBlocks:
                        with pytest.raises(pkv.PkvError) as e:
                            pkv.pkv_cow_block(h, r, idx)
                        assert e.value.code == pkv.PKV_ERR_OOM
                    else:
                        assert pkv.pkv_cow_block(h, r, idx) == want
            else:
                r = live.pop(rng.randrange(len(live)))
                ref.free(r)
                pkv.pkv_free(h, r)
            if i % 499 == 0:
                assert pkv.pkv_free_list(h) == ref.free_list
                for r in live[:6]:
                    t = pkv.pkv_request_table(h, r)
                    assert t == ref.table(r)
                    assert [pkv.pkv_block_refs(h, b) for b in t] == [ref.refs(b) for b in t]
        assert pkv.pkv_free_list(h) == ref.free_list
        for b in range(n):
            assert pkv.pkv_block_refs(h, b) == ref.refs(b)
    finally:
        pkv.pkv_allocator_destroy(h)


def test_fork_and_cow_errors(L):
    h = pkv.pkv_allocator_create(6, 16)
    try:
        prefix = pkv.pkv_alloc(h, -1, 1)
        pkv.pkv_alloc(h, 1, 1)
        pkv.pkv_attach_shared(h, 1, prefix)
        for fn, args, code in [(pkv.pkv_fork, (9, 2), pkv.PKV_ERR_NOT_FOUND),
                               (pkv.pkv_fork, (1, -1), pkv.PKV_ERR_EXISTS),
                               (pkv.pkv_cow_block, (1, 0), pkv.PKV_ERR_INVALID),   # pinned prefix
                               (pkv.pkv_cow_block, (1, 2), pkv.PKV_ERR_INVALID),   # past the table
                               (pkv.pkv_cow_block, (9, 0), pkv.PKV_ERR_NOT_FOUND),
                               (pkv.pkv_block_refs, (6,), pkv.PKV_ERR_INVALID)]:
            with pytest.raises(pkv.PkvError) as e:
                fn(h, *args)
            assert e.value.code == code, (fn, args)
        pkv.pkv_fork(h, 1, 2)
        assert pkv.pkv_request_table(h, 2) == prefix + [1]
        assert pkv.pkv_block_refs(h, 1) == 2 and pkv.pkv_block_refs(h, prefix[0]) == 1
        assert pkv.pkv_cow_block(h, 2, 1) == (1, 2)
        assert pkv.pkv_cow_block(h, 1, 1) is None
        pkv.pkv_free(h, 1)
        assert pkv.pkv_free_list(h) == [3, 4, 5, 1]
    finally:
        pkv.pkv_allocator_destroy(h)


def test_cache_stats_count_blocks_and_tail_waste(L):
    """Pool occupancy of the runtime: used + free = total, tail waste below one
    block per sequence, shared prefix blocks counted once."""
    import torch
    from paged_kv_cache_56_gb300.runtime import PagedKVCache
    c = PagedKVCache(2, 32, 4, 2, 64, 16, False, max_slots=4, max_blocks_per_seq=8, device="cpu")
    try:
        c.add_sequence(-1, 2)
        prefix = c.table(-1)
        c.seqs[-1].length = 32
        c.add_sequence(7, 3, shared_blocks=prefix)
        c.seqs[7].length = 2 * 16 + 40
        c.add_sequence(8, 1, shared_blocks=prefix)
        c.seqs[8].length = 2 * 16 + 1
        st = c.stats()
        assert st["blocks_total"] == 32 and st["blocks_used"] == 6 and st["blocks_free"] == 26
        assert st["blocks_referenced"] == 6 and st["sequences"] == 3
        assert st["tail_waste_tokens"] == (5 * 16 - 72) + (3 * 16 - 33)
    finally:
        c.close()


def test_missing_library_fails_loudly(tmp_path):
    """Without the built library the binding raises instead of falling back to
    anything else (there is no CPU path)."""
    import subprocess
    import sys
    code = ("import sys; sys.path.insert(0, {root!r});"
            "from paged_kv_cache_56_gb300 import pkv; pkv.LIB_PATH = {missing!r}; pkv._lib = None\n"
            "try:\n    pkv.lib()\nexcept RuntimeError as e:\n    print('raised', e)\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code.format(root=root, missing=str(tmp_path / "libpkv.so"))],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.startswith("raised"), (r.stdout, r.stderr)
