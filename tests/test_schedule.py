"""Host-side model of the persistent stream-K schedule, checked for the
properties the kernel relies on (no GPU).

The kernel walks each unit's items with the same rules: whole tiles
round-robin, then the unit's equal share of the split k-blocks from its last
tile back to its first.  A split tile's parts are added by the unit holding
its last k-block, after waiting for the lower units holding its earlier
k-blocks.  The model checks, over a sweep of tile counts, grid sizes and
k-block counts, that

* every k-block of every tile is computed exactly once;
* a unit holds at most one part that ends inside a tile (one partial-sum
  slot per unit), and it is that unit's first split item;
* the unit adding a tile's parts waits only on lower units, each of which
  publishes that part as its first split item (no cycle of waits, and with
  CTAs dispatched in index order no wait on a CTA that cannot start);
* no unit has an empty range.

The grid choice mirrors the library's planner: tiles < slots splits all
tiles over u = min(slots, ceil(tiles * k_blocks / 8)) units when u is at
least three times the tile count, or (single CTAs, compute-bound GEMMs)
when that takes 1536 k values or more off each unit (unless the GEMM is
memory-bound and its tiles already fill half the slots); more tiles than slots with a partial
last wave at most 4/5 full split the last two waves' tiles (slots + tiles %
slots) over all slots -- for quads (the plan for C rows off 16-byte
boundaries) only a last wave at most half full after two full waves.  `force` is the plan override that splits wherever
the schedule can.
"""
from __future__ import annotations

import itertools

import pytest

MIN_SPLIT_KB = 8
MIN_SAVED_K = 1536


def plan(tiles: int, slots: int, num_kb: int, memory_bound: bool = False, force: bool = False,
         quad: bool = False, single: bool = False, bk: int = 64):
    units, dp_tiles, sk_tiles = min(tiles, slots), tiles, 0
    tail = tiles % slots
    tail_rule = (2 * tail <= slots and tiles >= 2 * slots) if quad else 5 * tail <= 4 * slots
    if tiles < slots:
        u = min(slots, -(-tiles * num_kb // MIN_SPLIT_KB))
        saved_k = (num_kb - -(-tiles * num_kb // u)) * bk if u > tiles else 0
        pays = u >= 3 * tiles or (single and not memory_bound and saved_k >= MIN_SAVED_K)
        if u > tiles and (force or (pays and not (memory_bound and 2 * tiles >= slots))):
            units, dp_tiles, sk_tiles = u, 0, tiles
    elif tiles > slots and tail and num_kb > 1 and (force or tail_rule):
        sk_tiles = slots + tiles % slots
        dp_tiles = tiles - sk_tiles
    return units, dp_tiles, sk_tiles


def sk_begin(sk_work: int, units: int, u: int) -> int:
    return sk_work * u // units


def items(u: int, units: int, dp_tiles: int, sk_tiles: int, num_kb: int):
    """(tile, kb0, kb1, kind) in processing order; kinds as in the kernel."""
    out = []
    for t in range(u, dp_tiles, units):
        out.append((t, 0, num_kb, 0))
    sk_work = sk_tiles * num_kb
    beg, pos = sk_begin(sk_work, units, u), sk_begin(sk_work, units, u + 1)
    while pos > beg:
        t = (pos - 1) // num_kb
        ts = t * num_kb
        kb1 = pos - ts
        kb0 = beg - ts if beg > ts else 0
        pos = ts + kb0
        kind = 1 if kb1 < num_kb else (2 if kb0 > 0 else 0)
        out.append((dp_tiles + t, kb0, kb1, kind))
    return out


def first_part_unit(u: int, sk_tile: int, units: int, sk_work: int, num_kb: int) -> int:
    tile_start = sk_tile * num_kb
    v = u - 1
    while v > 0 and sk_begin(sk_work, units, v) > tile_start:
        v -= 1
    return v


CASES = [(t, g, k) for t, g, k in itertools.product(
    [1, 2, 3, 5, 17, 73, 74, 75, 100, 147, 148, 149, 160, 296, 300, 512],
    [1, 2, 7, 74, 148],
    [1, 2, 3, 7, 8, 9, 64, 65, 256])]


@pytest.mark.parametrize("mode", ["compute", "memory", "forced"])
@pytest.mark.parametrize("tiles,slots,num_kb", CASES)
def test_schedule_properties(tiles, slots, num_kb, mode):
    units, dp_tiles, sk_tiles = plan(tiles, slots, num_kb, mode == "memory", mode == "forced")
    assert units <= slots and dp_tiles + sk_tiles == tiles
    sk_work = sk_tiles * num_kb
    if sk_tiles:
        assert sk_work >= units
        for u in range(units):
            assert sk_begin(sk_work, units, u + 1) > sk_begin(sk_work, units, u)
    per_unit = [items(u, units, dp_tiles, sk_tiles, num_kb) for u in range(units)]
    cover = {}
    writers = {}  # tile -> units with a kind-1 part
    for u, its in enumerate(per_unit):
        kinds = [k for (_, _, _, k) in its]
        assert kinds.count(1) <= 1
        split = [it for it in its if it[0] >= dp_tiles]
        if 1 in kinds:
            assert split[0][3] == 1  # the first split item
        if 2 in kinds:
            assert its[-1][3] == 2 and kinds.count(2) == 1  # the last item
        for (t, kb0, kb1, kind) in its:
            assert 0 <= kb0 < kb1 <= num_kb
            for kb in range(kb0, kb1):
                assert (t, kb) not in cover
                cover[(t, kb)] = u
            if kind == 1:
                writers.setdefault(t, []).append(u)
    assert len(cover) == tiles * num_kb
    finished = set()
    for u, its in enumerate(per_unit):
        for (t, kb0, kb1, kind) in its:
            if kind == 2:
                v_lo = first_part_unit(u, t - dp_tiles, units, sk_work, num_kb)
                assert sorted(writers.get(t, [])) == list(range(v_lo, u))
                finished.add(t)
    # Every split tile that has writer parts is finished by exactly one unit.
    assert set(writers) <= finished
    for t in writers:
        assert t >= dp_tiles


def items_incremental(u: int, units: int, dp_tiles: int, sk_tiles: int, num_kb: int):
    """The kernel's form of the same walk: one division per unit for the
    first split tile, then one tile back per item."""
    out = [(t, 0, num_kb, 0) for t in range(u, dp_tiles, units)]
    sk_work = sk_tiles * num_kb
    beg, pos = sk_begin(sk_work, units, u), sk_begin(sk_work, units, u + 1)
    t = (pos - 1) // num_kb if pos > beg else 0
    while pos > beg:
        ts = t * num_kb
        kb1 = pos - ts
        kb0 = beg - ts if beg > ts else 0
        pos = ts + kb0
        out.append((dp_tiles + t, kb0, kb1, 1 if kb1 < num_kb else (2 if kb0 > 0 else 0)))
        t -= 1
    return out


@pytest.mark.parametrize("mode", ["compute", "forced"])
def test_incremental_split_walk_matches(mode):
    for tiles, slots, num_kb in CASES:
        units, dp_tiles, sk_tiles = plan(tiles, slots, num_kb, False, mode == "forced")
        for u in range(units):
            assert items_incremental(u, units, dp_tiles, sk_tiles, num_kb) == items(u, units, dp_tiles, sk_tiles, num_kb)


def test_balance_when_tiles_overflow_the_grid():
    # Equal shares: every unit's k-block count is within one tile's worth of
    # the mean (whole tiles) plus one k-block (split ranges).
    for tiles, slots, num_kb in [(256, 74, 64), (192, 74, 65), (512, 148, 64), (300, 148, 7)]:
        units, dp, sk = plan(tiles, slots, num_kb)
        work = [sum(kb1 - kb0 for (_, kb0, kb1, _) in items(u, units, dp, sk, num_kb)) for u in range(units)]
        assert max(work) - min(work) <= 1


def tile_coords(tile: int, m_tiles: int, n_tiles: int, group_m: int) -> tuple[int, int]:
    """The kernel's grouped tile order: group_m tile rows at a time, m
    fastest inside a group."""
    per_group = group_m * n_tiles
    g, i = divmod(tile, per_group)
    first = g * group_m
    gm = min(group_m, m_tiles - first)
    return first + i % gm, i // gm


@pytest.mark.parametrize("m_tiles,n_tiles", [(1, 1), (16, 16), (16, 12), (32, 32), (5, 7), (64, 1), (1, 64)])
@pytest.mark.parametrize("units", [1, 8, 76, 152])
def test_grouped_tile_order_is_a_bijection(m_tiles, n_tiles, units):
    gm = 1
    while (gm + 1) ** 2 <= units:
        gm += 1
    gm = min(gm, m_tiles)
    seen = {tile_coords(t, m_tiles, n_tiles, gm) for t in range(m_tiles * n_tiles)}
    assert seen == {(m, n) for m in range(m_tiles) for n in range(n_tiles)}
    if m_tiles == n_tiles == 32 and units == 76:
        # A wave of 76 tiles touches 8 rows of A panels and 10 columns of B.
        wave = {tile_coords(t, m_tiles, n_tiles, gm) for t in range(76)}
        assert len({m for m, _ in wave}) == 8 and len({n for _, n in wave}) == 10


def test_quad_split_rule_matches_the_measured_cases():
    # 36 quads: split only a last wave at most half full after >= 2 waves.
    assert plan(96, 36, 65, quad=True)[2] == 0      # 2.67 waves: whole tiles measured faster
    assert plan(48, 36, 32, quad=True)[2] == 0      # 1.33 waves: whole
    assert plan(384, 36, 64, quad=True)[2] == 0     # 10.67 waves: whole
    assert plan(120, 36, 63, quad=True)[2] == 36 + 120 % 36  # 3.33 waves: split measured 6% faster
    # Pairs keep the 4/5 rule.
    assert plan(96, 36, 65)[2] == 36 + 96 % 36
    # Forced splits ignore both rules; the schedule invariants hold either way.
    assert plan(96, 36, 65, quad=True, force=True)[2] == 36 + 96 % 36


def test_single_cta_split_rule_matches_the_measured_cases():
    # Single CTAs, M = N = 1024 (64 tiles on 152 SMs), 64-k blocks: the
    # split measured faster from K = 3072 on, slower at K = 2048.
    assert plan(64, 152, 32, single=True)[2] == 0          # K = 2048: 1152 k fewer per unit
    assert plan(64, 152, 48, single=True)[2] == 64         # K = 3072: 1728
    assert plan(64, 152, 64, single=True)[2] == 64         # K = 4096
    assert plan(64, 152, 128, single=True)[2] == 64        # K = 8192
    assert plan(64, 152, 16, single=True)[2] == 0          # 1024^3: u = 128 units of 8 k-blocks
    # Memory-bound shapes and CTA pairs keep the older rule.
    assert plan(64, 152, 64, single=True, memory_bound=True)[2] == 0
    assert plan(32, 76, 64)[2] == 0 and plan(48, 76, 64)[2] == 0 and plan(64, 76, 64)[2] == 0
    # The schedule invariants hold for the new splits too.
    for num_kb in (48, 64, 128):
        units, dp, sk = plan(64, 152, num_kb, single=True)
        seen = {}
        for u in range(units):
            for t, kb0, kb1, _ in items(u, units, dp, sk, num_kb):
                for kb in range(kb0, kb1):
                    assert (t, kb) not in seen
                    seen[(t, kb)] = u
        assert len(seen) == 64 * num_kb
