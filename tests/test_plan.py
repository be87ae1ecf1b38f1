"""Host work plan (mla_plan_units) on the CPU: the plan is a permutation of
the attend kernel's work units in its numbering, each CTA's list ascending,
and its busiest CTA within the list-scheduling bound; the planned entry
point rejects what it can check on the host.  No kernel runs here."""

import ctypes

import numpy as np
import pytest
import torch

import mla_decode_paged_gb300 as mla

NULL = ctypes.c_void_p(0)
P16 = ctypes.c_void_p(1 << 20)   # never dereferenced: each case below fails validation first


@pytest.fixture(scope="module")
def lib():
    mla.build()
    return mla.library()


def _units(lengths, qlen, heads, ns, st):
    """Per-unit token counts in the kernels' order: request-major, then
    split k (the split rule of mla_decode.h), then query-row group."""
    rows = qlen * heads
    groups = -(-rows // 48)
    out = []
    for L in lengths:
        L = max(int(L), 0)
        n = max(1, min(ns, -(-L // st)))
        b, m = divmod(L, n)
        for k in range(n):
            out += [b + (1 if k < m else 0)] * groups
    return out


def _split(plan):
    plan = plan.numpy()
    G = int(plan[0])
    off = plan[1:G + 2]
    ids = plan[G + 2:]
    return G, off, ids


CASES = [
    # lengths, qlen, heads, num_splits, split_tokens, G
    ([5000, 100, 8000, 1, 0, 4096], 1, 12, 7, 1167, 152),
    (list(range(1, 300)), 1, 12, 4, 64, 152),
    ([12000] * 32, 1, 96, 7, 4682, 152),             # two row groups of 48
    ([4000, 9000, 300] * 40, 4, 12, 5, 6543, 148),
    ([3] * 7, 8, 12, 31, 3992, 8),                   # fewer CTAs than units per request
    ([], 1, 12, 1, 16, 152),
]


@pytest.mark.parametrize("lengths,qlen,heads,ns,st,G", CASES)
def test_plan_is_a_permutation_in_kernel_numbering(lengths, qlen, heads, ns, st, G):
    plan = mla.plan_units(lengths, qlen, heads, ns, st, sm_count=G)
    units = _units(lengths, qlen, heads, ns, st)
    assert plan.dtype == torch.int32 and plan.numel() == 2 + G + len(units)
    g, off, ids = _split(plan)
    assert g == G
    assert off[0] == 0 and off[-1] == len(units) and np.all(np.diff(off) >= 0)
    assert sorted(ids.tolist()) == list(range(len(units)))
    for b in range(G):
        mine = ids[off[b]:off[b + 1]]
        assert np.all(np.diff(mine) > 0), "CTA %d's units are not ascending" % b


@pytest.mark.parametrize("lengths,qlen,heads,ns,st,G", CASES[:5])
def test_plan_balance_within_list_scheduling_bound(lengths, qlen, heads, ns, st, G):
    """Greedy assignment to the least loaded CTA keeps the busiest CTA within
    mean + the largest unit (Graham's bound); longest-first is never worse
    than round robin on these length mixes."""
    units = _units(lengths, qlen, heads, ns, st)
    cost = [-(-c // 128) + (0.5 if c else 0.2) for c in units]
    g, off, ids = _split(mla.plan_units(lengths, qlen, heads, ns, st, sm_count=G))
    load = [sum(cost[i] for i in ids[off[b]:off[b + 1]]) for b in range(G)]
    assert max(load) <= sum(cost) / G + max(cost) + 1e-9
    rr = [sum(cost[u] for u in range(b, len(cost), G)) for b in range(G)]
    assert max(load) <= max(rr) + 1e-9


def test_plan_example_by_hand():
    """Three requests of 256, 128 and 1 tokens, one split each, two CTAs:
    costs 2.5, 1.5, 1.5 -> unit 0 alone on CTA 0, units 1 and 2 on CTA 1."""
    plan = mla.plan_units([256, 128, 1], 1, 12, 1, 4096, sm_count=2)
    assert plan.tolist() == [2, 0, 1, 3, 0, 1, 2]


def test_plan_size_query_and_errors(lib):
    lens = torch.tensor([100, 200], dtype=torch.int32)
    lp = ctypes.c_void_p(lens.data_ptr())
    n = lib.mla_plan_units(2, 1, 12, lp, 4, 64, 10, None, 0)
    assert n == 2 + 10 + (2 + 4)
    buf = torch.empty(n - 1, dtype=torch.int32)
    assert lib.mla_plan_units(2, 1, 12, lp, 4, 64, 10, ctypes.c_void_p(buf.data_ptr()), n - 1) == mla.MLA_ERR_INVALID
    assert b"too small" in lib.mla_last_error()
    for bad in [(2, 0, 12, lp, 4, 64), (2, 1, 0, lp, 4, 64), (2, 1, 12, lp, 0, 64), (2, 1, 12, lp, 4, 0),
                (2, 1, 12, NULL, 4, 64), (-1, 1, 12, lp, 4, 64)]:
        assert lib.mla_plan_units(*bad, 10, None, 0) == mla.MLA_ERR_INVALID


def _attend_planned(lib, plan, plan_len, page_size=1, last=NULL):
    return lib.mla_decode_attend_planned(P16, 12 * 576, P16, 128, P16, 10, P16, last, page_size, 2, 1, 12, 0.1, 1.0,
                                         4, 16, P16, P16, 0, plan, plan_len, NULL)


def test_planned_attend_rejects_short_or_misaligned_plans(lib):
    assert _attend_planned(lib, P16, 2) == mla.MLA_ERR_INVALID
    assert b"plan" in lib.mla_last_error()
    assert _attend_planned(lib, ctypes.c_void_p((1 << 20) + 2), 20) == mla.MLA_ERR_INVALID
    assert b"plan" in lib.mla_last_error()


def test_planned_attend_with_warp_mma_kernel_is_unsupported(lib, monkeypatch):
    monkeypatch.setenv("MLA_ATTEND_KERNEL", "mma")
    assert _attend_planned(lib, P16, 20) == mla.MLA_ERR_UNSUPPORTED
    assert b"work plan" in lib.mla_last_error()
