"""GPU checks of the host work plan (mla_decode_attend_planned): with a plan
the attend partials are bit-identical to the round-robin launch and match
the oracle; plans that do not fit the launch are flagged, not faulted."""

import numpy as np
import pytest
import torch

import mla_decode_paged_gb300 as mla
from mla_decode_paged_gb300 import workloads as W
from oracle import mla_oracle as O
from tests._bits import bf16_bits, i32, oracle_args, u8
from tests.parity import assert_bf16_close, assert_lse_close

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.build()
    mla.device_status()
    yield


def _dev(inp):
    out = W.Inputs(inp.spec, *(getattr(inp, f).to(DEV) for f in
                               ("q", "kv", "pages", "indptr", "lengths", "w_uv", "gate")),
                   inp.scale, inp.kv_scale)
    for k, v in inp.extra.items():
        out.extra[k] = v.to(DEV) if torch.is_tensor(v) else v
    return out


def _attend(inp, ns, st, plan=None, **kw):
    if inp.extra.get("page_size", 1) > 1:
        kw.update(page_size=inp.extra["page_size"], last_page_len=inp.extra["last_page_len"])
    o, lse = mla.attend(inp.q, inp.kv, inp.pages, inp.indptr, inp.scale, inp.kv_scale, ns, st, heads=inp.heads,
                        qlen=inp.qlen, plan=plan, **kw)
    torch.cuda.synchronize()
    return o, lse


def _same(a, b):
    """Partials equal bit for bit wherever the split is used (finite lse)."""
    (o1, l1), (o2, l2) = a, b
    used = torch.isfinite(l1)
    assert torch.equal(torch.isfinite(l2), used)
    assert torch.equal(l1[used], l2[used])
    assert torch.equal(o1[used].view(torch.int16), o2[used].view(torch.int16))


def _plan(inp_lengths, inp, ns, st):
    return mla.plan_units(inp_lengths.cpu(), inp.qlen, inp.heads, ns, st).to(DEV)


@pytest.mark.parametrize("idx,lengths,ns,st", [
    (1, [1, 17, 128, 129, 300, 1000], 4, 64),
    (2, [257, 64, 700], 8, 50),
    (3, [300, 129], 3, 7),
    (4, [0, 5, 200, 0, 333], 4, 64),
])
def test_planned_small_workloads_match_oracle_and_round_robin(idx, lengths, ns, st):
    inp_cpu = W.make_inputs(idx, "cpu", lengths=lengths)
    inp = _dev(inp_cpu)
    plan = _plan(inp_cpu.lengths, inp, ns, st)
    got = _attend(inp, ns, st, plan)
    _same(got, _attend(inp, ns, st))
    ro, rl = O.attend_splits(**oracle_args(inp_cpu), num_splits=ns, split_tokens=st)
    assert_lse_close(got[1], rl, "planned partial lse")
    assert_bf16_close(got[0], ro, "planned partial o", mask=np.isfinite(rl))
    assert mla.device_status() == 0


@pytest.mark.parametrize("idx", [1, 2, 3, 4])
def test_planned_full_size_workloads(idx):
    """The launch configuration the benchmark times: bit-identical partials,
    merged output checked against the oracle on sampled requests."""
    inp = W.make_inputs(idx, DEV)
    ns, st = mla.choose_splits(inp.spec.requests, inp.qlen, inp.heads, lengths=inp.lengths.cpu())
    plan = _plan(inp.lengths, inp, ns, st)
    got = _attend(inp, ns, st, plan)
    _same(got, _attend(inp, ns, st))
    latent, lse_m = mla.merge(*got)
    torch.cuda.synchronize()
    lens = i32(inp.lengths)
    rng = np.random.default_rng(idx)
    reqs = sorted(set([int(lens.argmax())] + [int(x) for x in rng.choice(len(lens), 2, replace=False)]))
    a = dict(q_bits=bf16_bits(inp.q), kv_codes=u8(inp.kv), pages=i32(inp.pages), indptr=i32(inp.indptr),
             scale=inp.scale, kv_scale=inp.kv_scale, heads=inp.heads, qlen=inp.qlen)
    rlat, rlse = O.attend(**a, requests=reqs)
    rows = np.concatenate([np.arange(r * inp.qlen, (r + 1) * inp.qlen) for r in reqs])
    assert_lse_close(lse_m[rows], rlse[rows], "planned lse (sampled)")
    assert_bf16_close(latent[rows], rlat[rows], "planned latent (sampled)")
    assert mla.device_status() == 0


def test_planned_block_tables_causal_identical():
    inp = W.make_block_inputs(2, DEV, page_size=16)
    ns, st = mla.choose_splits(inp.spec.requests, inp.qlen, inp.heads, lengths=inp.lengths.cpu())
    plan = _plan(inp.lengths, inp, ns, st)
    _same(_attend(inp, ns, st, plan, causal=True), _attend(inp, ns, st, causal=True))
    assert mla.device_status() == 0


def _small():
    inp_cpu = W.make_inputs(1, "cpu", lengths=[1, 17, 128, 129, 300, 1000, 0, 640])
    inp = _dev(inp_cpu)
    ns, st = 4, 64
    return inp, ns, st, mla.plan_units(inp_cpu.lengths, inp.qlen, inp.heads, ns, st)


def test_plan_for_another_grid_is_flagged():
    inp, ns, st, plan = _small()
    bad = plan.clone()
    bad[0] += 1
    _attend(inp, ns, st, bad.to(DEV))
    assert mla.device_status() & mla.DEV_BAD_PLAN
    assert mla.device_status() == 0


def test_plan_offsets_outside_the_buffer_are_flagged():
    inp, ns, st, plan = _small()
    G = int(plan[0])
    bad = plan.clone()
    bad[1 + G] = plan.numel()        # the last CTA's list runs past the ids
    _attend(inp, ns, st, bad.to(DEV))
    assert mla.device_status() & mla.DEV_BAD_PLAN
    assert mla.device_status() == 0


def test_plan_with_decreasing_ids_is_flagged():
    inp, ns, st, plan = _small()
    G = int(plan[0])
    U = plan.numel() - 2 - G
    assert U <= G
    # CTA 0 takes units 1 then 0 (decreasing), CTA b > 0 takes unit b + 1
    counts = [2] + [1] * (U - 2) + [0] * (G - U + 1)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    ids = np.array([1, 0] + list(range(2, U)), dtype=np.int32)
    bad = torch.from_numpy(np.concatenate([[G], off, ids]).astype(np.int32))
    assert bad.numel() == plan.numel()
    _attend(inp, ns, st, bad.to(DEV))
    assert mla.device_status() & mla.DEV_BAD_PLAN
    assert mla.device_status() == 0


def test_plan_id_past_the_last_unit_ends_that_list():
    """An id beyond the units ends its CTA's list without a flag; every other
    unit's partial is still the round-robin one."""
    inp, ns, st, plan = _small()
    G = int(plan[0])
    off = plan[1:G + 2]
    b = int(np.argmax((off[1:] - off[:-1]).numpy() >= 1))
    last = G + 2 + int(off[b + 1]) - 1
    dropped = int(plan[last])
    bad = plan.clone()
    bad[last] = 1 << 30
    o, lse = _attend(inp, ns, st, bad.to(DEV))
    assert mla.device_status() == 0
    ro, rl = _attend(inp, ns, st)
    # unit ids are (request, split) pairs request-major (one row group here)
    lens = i32(inp.lengths)
    pairs = [(r, k) for r, L in enumerate(lens) for k in range(max(1, min(ns, -(-int(L) // st))))]
    r_d, k_d = pairs[dropped]
    keep = torch.isfinite(rl)
    keep[k_d, r_d * inp.qlen:(r_d + 1) * inp.qlen] = False
    assert torch.equal(lse[keep], rl[keep])
    assert torch.equal(o[keep].view(torch.int16), ro[keep].view(torch.int16))
