"""Host-side checks of the decode kernel's staged-tile layout (no GPU).

The decode kernel stages 16-token K/V tiles of 128- or 256-byte rows with a
128-byte-swizzled tensor copy: byte `off` of row r of a tile sits in the
2048-byte slab off // 128, at 16-byte chunk position ((off % 128) // 16) ^ (r % 8).
Lane (g = lane // 4, t = lane % 4) of a warp reads its K run of token rows g and
g + 8 and its V run of token rows 2t, 2t+1, 2t+8, 2t+9; at bf16 d = 128 the runs
are split over the two 128-byte halves of a row. These tests restate that
arithmetic and check what the layout promises:

* the K runs of lanes t = 0..3 cover the row's bytes exactly once, and so do the
  V runs of lanes g = 0..7 (each dim enters QK and PV exactly once);
* the output scatter puts every dim of every lane's V run in its own place;
* every 16-byte shared-memory load of a quarter-warp (8 lanes) hits 8 different
  16-byte bank groups (no bank conflict), where the unswizzled linear layout
  conflicted.
"""

import itertools

import pytest

# (head_dim, bytes per element, lanes' runs split over the row's halves)
CONFIGS = [(128, 1, False), (128, 2, True), (64, 2, False)]


def k_run_bytes(d, e):  # bytes of a row one lane t reads for QK
    return d // 4 * e


def v_run_bytes(d, e):  # bytes of a row one lane g reads for PV
    return d // 8 * e


def k_chunk(nb, halves, t, c):
    return (c >> 1) * 128 + t * (nb // 2) + (c & 1) * 16 if halves else t * nb + c * 16


def v_chunk(nb, halves, g, c):
    return c * 128 + g * (nb // 2) if halves else g * nb + c * 16


def swizzled(off, r):
    """Shared-memory byte offset of row r's byte `off` within a staged tile."""
    return (off >> 7) * 2048 + r * 128 + ((((off >> 4) & 7) ^ (r & 7)) << 4) + (off & 15)


def linear(off, r, row):
    return r * row + off


def bank_group(addr):  # 16-byte unit of the 128-byte bank window
    return (addr >> 4) & 7


@pytest.mark.parametrize("d,e,halves", CONFIGS)
def test_runs_cover_each_row_byte_once(d, e, halves):
    row = d * e
    kb, vb = k_run_bytes(d, e), v_run_bytes(d, e)
    k_bytes = sorted(k_chunk(kb, halves, t, c) + i for t in range(4) for c in range(kb // 16) for i in range(16))
    v_bytes = sorted(v_chunk(vb, halves, g, c) + i for g in range(8) for c in range(vb // 16) for i in range(16))
    assert k_bytes == list(range(row))
    assert v_bytes == list(range(row))


@pytest.mark.parametrize("d,e,halves", CONFIGS)
def test_output_scatter_matches_v_runs(d, e, halves):
    """m-tile m's rows g and g + 8 hold the two dims of word m of lane g's V
    run; the output scatter must name exactly those dims."""
    vb = v_run_bytes(d, e)
    for g in range(8):
        run_dims = [(v_chunk(vb, halves, g, c) + i) // e for c in range(vb // 16) for i in range(0, 16, e)]
        if e == 2:  # bf16: word j = dims (2j, 2j+1) of the run, one m-tile per word
            for m in range(d // 16):
                d0 = (m >> 2) * (d // 2) + g * 8 + 2 * (m & 3) if halves else g * (d // 8) + 2 * m
                assert (d0, d0 + 1) == (run_dims[2 * m], run_dims[2 * m + 1])
        else:  # int8: the run is contiguous and the scatter is the plain one
            assert run_dims == list(range(g * (d // 8), (g + 1) * (d // 8)))


def _quarter_warp_groups(addr_of_lane):
    """Bank groups hit by each quarter-warp's 16-byte loads."""
    out = []
    for qw in range(4):
        lanes = range(8 * qw, 8 * qw + 8)
        out.append([bank_group(addr_of_lane(lane)) for lane in lanes])
    return out


@pytest.mark.parametrize("d,e,halves", CONFIGS)
def test_swizzled_loads_are_conflict_free(d, e, halves):
    kb, vb = k_run_bytes(d, e), v_run_bytes(d, e)
    # K: rows g and g + 8, every 16-byte chunk of the run
    for dr, c in itertools.product((0, 8), range(kb // 16)):
        groups = _quarter_warp_groups(lambda lane: swizzled(k_chunk(kb, halves, lane % 4, c), lane // 4 + dr))
        assert all(len(set(gs)) == 8 for gs in groups), (d, e, "K", dr, c, groups)
    # V: rows 2t, 2t+1, 2t+8, 2t+9
    for dr, c in itertools.product((0, 1, 8, 9), range(vb // 16)):
        groups = _quarter_warp_groups(lambda lane: swizzled(v_chunk(vb, halves, lane // 4, c), 2 * (lane % 4) + dr))
        assert all(len(set(gs)) == 8 for gs in groups), (d, e, "V", dr, c, groups)


@pytest.mark.parametrize("d,e", [(128, 1), (128, 2)])
def test_linear_layout_conflicted(d, e):
    """The unswizzled layout the tensor copies replaced: V loads of a
    quarter-warp fall into at most 2-4 bank groups (what ncu counted)."""
    row, vb = d * e, v_run_bytes(d, e)
    groups = _quarter_warp_groups(lambda lane: linear(v_chunk(vb, False, lane // 4, 0), 2 * (lane % 4), row))
    assert max(len(set(gs)) for gs in groups) <= 4


def test_tensor_copy_coordinates_are_16_byte_aligned():
    """Each tile's boxes start at x = 0 or 128 bytes of the row (the copy's
    innermost coordinate must be a multiple of 16 bytes)."""
    for row in (128, 256):
        xs = [h * 128 for h in range(row // 128)]
        assert all(x % 16 == 0 and x + 128 <= row for x in xs)
