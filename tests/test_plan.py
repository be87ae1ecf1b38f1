"""Host work plan (mla_plan_units) on the CPU: every request's tokens are
cut into consecutive splits at tile boundaries, each split once per row
group, the row groups of a request on adjacent CTAs with the same items,
at most num_splits splits per request, and the busiest CTA within one tile
of the mean (or of the longest request's share per split); the planned entry point rejects what it can check on the host.
No kernel runs here."""

import ctypes

import numpy as np
import pytest
import torch

import mla_decode_paged_gb300 as mla
from tests import _plan

NULL = ctypes.c_void_p(0)
P16 = ctypes.c_void_p(1 << 20)   # never dereferenced: each case below fails validation first
TILE, EMPTY = 10, 2    # the planner's cost model, tenths of a 128-token tile


@pytest.fixture(scope="module")
def lib():
    mla.build()
    return mla.library()


def _groups(qlen, heads):
    return -(-qlen * heads // 48)


def _piece(qlen, heads):
    """The planner's fixed cost of a split for the CTA's query-row tile
    (4 tiles at 48 rows, 3 at 32, half a tile at 16)."""
    rows = qlen * heads
    g = -(-rows // 48)
    nq = -(-(-(-rows // g)) // 16) * 16
    return 40 if nq >= 48 else 30 if nq >= 32 else 5


def _cost(count, piece=5):
    return (-(-count // 128)) * TILE + piece if count > 0 else EMPTY


CASES = [
    # lengths, qlen, heads, num_splits, G
    ([5000, 100, 8000, 1, 0, 4096], 1, 12, 7, 152),
    (list(range(1, 300)), 1, 12, 4, 152),
    ([12000] * 32, 1, 96, 7, 152),              # two row groups of 48
    ([4000, 9000, 300] * 40, 4, 12, 5, 148),
    ([3] * 7, 8, 12, 31, 8),
    ([], 1, 12, 1, 152),
    ([70000, 10, 10, 10], 1, 12, 2, 152),       # num_splits binds
]


@pytest.mark.parametrize("lengths,qlen,heads,ns,G", CASES)
def test_plan_structure(lengths, qlen, heads, ns, G):
    plan, used = mla.plan_units(lengths, qlen, heads, ns, sm_count=G)
    g = _groups(qlen, heads)
    Gp, off, it = _plan.items(plan)
    assert Gp == G and plan.dtype == torch.int32
    assert plan.numel() == 2 + G + _plan.ITEM_WORDS * (it.shape[0] + G)
    assert off[0] == 0 and off[-1] == it.shape[0] and np.all(np.diff(off) >= 0)
    V = G // g
    for b in range(G):
        mine = it[off[b]:off[b + 1]]
        if b >= V * g:
            assert mine.shape[0] == 0
            continue
        assert np.all(mine[:, 3] == b % g)                     # row group of the CTA
        twin = it[off[b - b % g]:off[b - b % g + 1]]            # group 0 of the same virtual CTA
        assert np.array_equal(np.delete(mine, 3, axis=1), np.delete(twin, 3, axis=1))
    for grp in range(g):
        rg = _plan.ranges(plan, len(lengths), grp)
        for L, cuts in zip(lengths, rg):
            L = max(L, 0)
            assert cuts[0][0] == 0 and cuts[-1][1] == L
            assert all(a[1] == b[0] for a, b in zip(cuts, cuts[1:]))
            assert all(s % 128 == 0 for s, _ in cuts)
            assert all(e > s for s, e in cuts) or (L == 0 and cuts == [(0, 0)])
            assert len(cuts) <= ns
    assert used == max([len(c) for c in _plan.ranges(plan, len(lengths))] or [1])


@pytest.mark.parametrize("lengths,qlen,heads,ns,G", CASES[:6])
def test_plan_balance_within_a_tile_of_the_mean(lengths, qlen, heads, ns, G):
    """The budget is the smallest that fits the grid within num_splits
    splits per request, so every virtual CTA but the last ends within a tile
    and a split share of it: the busiest CTA is within that of the larger of
    the mean and the longest request's share per split."""
    plan, _ = mla.plan_units(lengths, qlen, heads, ns, sm_count=G)
    g = _groups(qlen, heads)
    V = G // g
    _, off, it = _plan.items(plan)
    piece = _piece(qlen, heads)
    loads = [sum(_cost(c, piece) for c in it[off[v * g]:off[v * g + 1], 5]) for v in range(V)]
    per_split = max([-(-(-(-L // 128)) // ns) * TILE + piece for L in lengths if L > 0] or [0])
    assert max(loads) <= max(sum(loads) / (V - 1), per_split) + TILE + piece


@pytest.mark.parametrize("lengths,qlen,heads,mn,ns,G", [
    ([4096, 30000, 9000, 700, 0, 129] * 20, 4, 12, 8, 32, 152),   # the speculative workload's kind of cut
    (list(range(1, 3000, 37)), 1, 12, 4, 16, 152),
    ([12000] * 32, 1, 96, 8, 32, 152),                           # two row groups
    ([1000, 128, 5], 8, 12, 8, 8, 16),                           # fewer tiles than min_splits
])
def test_plan_min_splits(lengths, qlen, heads, mn, ns, G):
    """mla_plan_units_ex: every request gets at least min(min_splits, its
    tiles) splits (num_splits allowing) and at most num_splits; the cuts stay
    tile-aligned and cover the tokens; the busiest CTA stays within a few
    pieces of the mean."""
    plan, used = mla.plan_units(lengths, qlen, heads, ns, sm_count=G, min_splits=mn)
    g = _groups(qlen, heads)
    for grp in range(g):
        for L, cuts in zip(lengths, _plan.ranges(plan, len(lengths), grp)):
            tiles = -(-max(L, 0) // 128)
            assert cuts[0][0] == 0 and cuts[-1][1] == max(L, 0)
            assert all(a[1] == b[0] for a, b in zip(cuts, cuts[1:])) and all(s % 128 == 0 for s, _ in cuts)
            assert len(cuts) <= ns
            if tiles:
                assert len(cuts) >= min(mn, tiles, ns)
    V = G // g
    _, off, it = _plan.items(plan)
    piece = _piece(qlen, heads)
    loads = [sum(_cost(c, piece) for c in it[off[v * g]:off[v * g + 1], 5]) for v in range(V)]
    cap = max(-(-(-(-max(lengths) // 128)) // mn), 1) if lengths else 1
    assert max(loads) <= sum(loads) / (V - 1) + cap * TILE + 2 * piece
    assert used == max(len(c) for c in _plan.ranges(plan, len(lengths)))


def test_plan_min_splits_one_is_the_plain_plan(lib):
    lens = [5000, 100, 8000, 1, 0, 4096]
    a, ua = mla.plan_units(lens, 1, 12, 7, sm_count=152)
    b, ub = mla.plan_units(lens, 1, 12, 7, sm_count=152, min_splits=1)
    assert torch.equal(a, b) and ua == ub
    lt = torch.tensor(lens, dtype=torch.int32)
    lp = ctypes.c_void_p(lt.data_ptr())
    n = lib.mla_plan_units(len(lens), 1, 12, lp, 7, 152, None, 0, None)
    assert n == a.numel()
    for bad in (0, 8):   # min_splits outside 1..num_splits
        assert lib.mla_plan_units_ex(len(lens), 1, 12, lp, bad, 7, 152, None, 0, None) == mla.MLA_ERR_INVALID
        assert b"min_splits" in lib.mla_last_error()


def test_plan_by_hand_without_cuts():
    """[256, 128, 1] tokens on 2 CTAs: costs 25, 15, 15; the smallest budget
    that fits is 30 (request 0 alone, then requests 1 and 2); then each
    CTA's first item again."""
    plan, used = mla.plan_units([256, 128, 1], 1, 12, 4, sm_count=2)
    one = 1 << 9
    assert plan.tolist() == [2, 0, 1, 3, 0, one, 0, 256, 1, one, 0, 128, 2, one, 0, 1,
                             0, one, 0, 256, 1, one, 0, 128]
    assert used == 1


def test_plan_by_hand_with_cuts():
    """1000 tokens (8 tiles) on 4 CTAs: budget 25 gives four splits of two
    tiles; with at most 3 splits the budget grows to 35 (3, 3, 2 tiles)."""
    plan, used = mla.plan_units([1000], 1, 12, 4, sm_count=4)
    assert used == 4 and _plan.ranges(plan, 1) == [[(0, 256), (256, 512), (512, 768), (768, 1000)]]
    plan, used = mla.plan_units([1000], 1, 12, 3, sm_count=4)
    assert used == 3 and _plan.ranges(plan, 1) == [[(0, 384), (384, 768), (768, 1000)]]
    _, off, _ = _plan.items(plan)
    assert off.tolist() == [0, 1, 2, 3, 3]


def test_plan_size_query_and_errors(lib):
    lens = torch.tensor([100, 200], dtype=torch.int32)
    lp = ctypes.c_void_p(lens.data_ptr())
    used = ctypes.c_int(0)
    n = lib.mla_plan_units(2, 1, 12, lp, 4, 10, None, 0, ctypes.byref(used))
    assert n == 2 + 10 + 4 * (3 + 10) and used.value == 2   # the 2-tile request is cut in two; 10 first-item copies
    buf = torch.empty(n - 1, dtype=torch.int32)
    assert lib.mla_plan_units(2, 1, 12, lp, 4, 10, ctypes.c_void_p(buf.data_ptr()), n - 1, None) == mla.MLA_ERR_INVALID
    assert b"too small" in lib.mla_last_error()
    for bad in [(2, 0, 12, lp, 4), (2, 1, 0, lp, 4), (2, 1, 12, lp, 0), (2, 1, 12, lp, 257),
                (2, 1, 12, NULL, 4), (-1, 1, 12, lp, 4)]:
        assert lib.mla_plan_units(*bad, 10, None, 0, None) == mla.MLA_ERR_INVALID
    assert lib.mla_plan_units(2, 1, 12, lp, 4, 65537, None, 0, None) == mla.MLA_ERR_INVALID
    assert b"sm_count" in lib.mla_last_error()
    # two row groups need at least two CTAs
    assert lib.mla_plan_units(2, 1, 96, lp, 4, 1, None, 0, None) == mla.MLA_ERR_UNSUPPORTED


def _attend_planned(lib, plan, plan_len, page_size=1, last=NULL, q_scale=1.0):
    return lib.mla_decode_attend_planned(P16, 12 * 576, P16, 128, P16, 10, P16, last, page_size, 2, 1, 12, 0.1, 1.0,
                                         q_scale, 4, 16, P16, P16, 0, plan, plan_len, NULL)


def test_planned_attend_rejects_short_or_misaligned_plans(lib):
    assert _attend_planned(lib, P16, 2) == mla.MLA_ERR_INVALID
    assert b"plan" in lib.mla_last_error()
    assert _attend_planned(lib, ctypes.c_void_p((1 << 20) + 2), 20) == mla.MLA_ERR_INVALID
    assert b"plan" in lib.mla_last_error()


def test_planned_attend_rejects_a_non_finite_q_scale(lib):
    assert _attend_planned(lib, P16, 20, q_scale=float("nan")) == mla.MLA_ERR_INVALID
    assert b"non-finite" in lib.mla_last_error()
