"""GPU checks of the balanced work plan (mla_decode_attend_planned): each
split's partial matches the oracle over the plan's token range, the merged
result matches the unsplit oracle, and plans that do not fit the launch are
flagged, not faulted."""

import numpy as np
import pytest
import torch

import mla_decode_paged_gb300 as mla
from mla_decode_paged_gb300 import workloads as W
from oracle import mla_oracle as O
from tests import _full as F
from tests import _plan
from tests._bits import bf16_bits, i32, oracle_args, u8
from tests.parity import assert_bf16_close, assert_lse_close, to_f64

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


def _attend(inp, ns, plan=None, st=64, **kw):
    if inp.extra.get("page_size", 1) > 1:
        kw.update(page_size=inp.extra["page_size"], last_page_len=inp.extra["last_page_len"])
    o, lse = mla.attend(inp.q, inp.kv, inp.pages, inp.indptr, inp.scale, inp.kv_scale, ns, st, heads=inp.heads,
                        qlen=inp.qlen, plan=None if plan is None else plan.to(DEV), **kw)
    torch.cuda.synchronize()
    return o, lse


def _block_args(inp_cpu):
    if inp_cpu.extra.get("page_size", 1) > 1:
        return dict(page_size=inp_cpu.extra["page_size"], last_page_len=i32(inp_cpu.extra["last_page_len"]))
    return {}


def _check_against_oracle(inp_cpu, o, lse, plan, ns, **kw):
    R = len(i32(inp_cpu.lengths))
    groups = -(-inp_cpu.qlen * inp_cpu.heads // 48)
    rg = _plan.ranges(plan, R, 0)
    for g in range(1, groups):
        assert _plan.ranges(plan, R, g) == rg
    a = oracle_args(inp_cpu)
    ro, rl = O.attend_splits(**a, num_splits=ns, split_tokens=1, ranges=rg, **_block_args(inp_cpu), **kw)
    assert_lse_close(lse, rl, "planned partial lse")
    assert_bf16_close(o, ro, "planned partial o", mask=np.isfinite(rl))
    latent, lse_m = mla.merge(o, lse)
    torch.cuda.synchronize()
    rlat, rlse = O.attend(**a, **_block_args(inp_cpu), **kw)
    assert_lse_close(lse_m, rlse, "planned merged lse")
    assert_bf16_close(latent, rlat, "planned latent")


@pytest.mark.parametrize("idx,lengths,ns", [
    (1, [1, 17, 128, 129, 300, 1000], 4),
    (2, [257, 64, 700], 8),
    (3, [300, 129], 3),                 # two row groups of 48
    (4, [0, 5, 200, 0, 333], 4),
    (1, [5000, 3, 40], 2),              # num_splits binds
    (4, [0, 0, 0], 3),                  # every request empty: lse -inf, latent 0
])
def test_planned_small_workloads_match_oracle(idx, lengths, ns):
    inp_cpu = W.make_inputs(idx, "cpu", lengths=lengths)
    inp = _dev(inp_cpu)
    plan, used = mla.plan_units(inp_cpu.lengths, inp.qlen, inp.heads, ns)
    assert used <= ns
    o, lse = _attend(inp, ns, plan)
    _check_against_oracle(inp_cpu, o, lse, plan, ns)
    assert mla.device_status() == 0


@pytest.mark.parametrize("idx,lengths,mn,ns", [
    (2, [4096, 700, 2000, 129, 0], 8, 32),   # the speculative workload's 8-32 partials
    (3, [1500, 300], 4, 8),                  # two row groups of 48
    (1, [1, 17, 128, 129, 300, 1000], 3, 4),
])
def test_min_splits_plans_match_oracle(idx, lengths, mn, ns):
    """mla_plan_units_ex: requests cut into at least min_splits splits (as
    their tiles allow); every split's partials and the merged rows against
    the oracle."""
    inp_cpu = W.make_inputs(idx, "cpu", lengths=lengths)
    inp = _dev(inp_cpu)
    plan, used = mla.plan_units(inp_cpu.lengths, inp.qlen, inp.heads, ns, min_splits=mn)
    assert used <= ns
    for L, cuts in zip(lengths, _plan.ranges(plan, len(lengths))):
        assert len(cuts) >= min(mn, -(-L // 128)) or L == 0
    o, lse = _attend(inp, ns, plan)
    _check_against_oracle(inp_cpu, o, lse, plan, ns)
    assert mla.device_status() == 0


def test_min_splits_plan_causal_block_tables_match_oracle():
    """A minimum-splits plan with the causal mask over a block-table cache
    (page size 16): consecutive splits of one request on one CTA."""
    inp_cpu = W.make_block_inputs(2, "cpu", page_size=16, lengths=[2, 3, 257, 1400, 700])
    inp = _dev(inp_cpu)
    plan, used = mla.plan_units(inp_cpu.lengths, inp.qlen, inp.heads, 16, min_splits=6)
    o, lse = _attend(inp, 16, plan, causal=True)
    _check_against_oracle(inp_cpu, o, lse, plan, 16, causal=True)
    assert mla.device_status() == 0


def test_min_splits_plan_full_size_speculative_workload(capsys):
    """The speculative workload cut into 8-32 partials per request by a
    balanced plan (the benchmark's stated cut with a plan): every row."""
    inp = W.make_inputs(2, DEV)
    plan, used = mla.plan_units(inp.lengths.cpu(), inp.qlen, inp.heads, 32, min_splits=8)
    cuts = _plan.ranges(plan, inp.spec.requests)
    assert min(len(c) for c in cuts) >= 8 and used <= 32
    latent, lse_m = mla.merge(*_attend(inp, used, plan))
    torch.cuda.synchronize()
    ref = F.reference(("plain", 2), inp)
    F.check_every_row("%s, plan with 8-32 partials" % inp.spec.name, ref, latent, lse_m, capsys=capsys)
    assert mla.device_status() == 0


def test_planned_causal_block_tables_match_oracle():
    inp_cpu = W.make_block_inputs(2, "cpu", page_size=16, lengths=[2, 3, 257, 700])
    inp = _dev(inp_cpu)
    plan, _ = mla.plan_units(inp_cpu.lengths, inp.qlen, inp.heads, 4)
    o, lse = _attend(inp, 4, plan, causal=True)
    _check_against_oracle(inp_cpu, o, lse, plan, 4, causal=True)
    assert mla.device_status() == 0


def test_planned_fp8_query_matches_oracle():
    inp_cpu = W.make_inputs(1, "cpu", lengths=[1, 17, 128, 129, 300, 1000])
    inp = _dev(inp_cpu)
    q8 = (inp_cpu.q.float() * 4).to(torch.float8_e4m3fn)     # codes of q * 4, read with q_scale 1/4
    plan, _ = mla.plan_units(inp_cpu.lengths, inp.qlen, inp.heads, 4)
    o, lse = mla.attend(q8.to(DEV), inp.kv, inp.pages, inp.indptr, inp.scale, inp.kv_scale, 4, 64, heads=inp.heads,
                        q_scale=0.25, plan=plan.to(DEV))
    latent, lse_m = mla.merge(o, lse)
    torch.cuda.synchronize()
    a = dict(oracle_args(inp_cpu), q_bits=u8(q8.view(torch.uint8)), scale=inp.scale * 0.25)
    rlat, rlse = O.attend(**a, q_fp8=True)
    assert_lse_close(lse_m, rlse, "planned fp8-query lse")
    assert_bf16_close(latent, rlat, "planned fp8-query latent")
    assert mla.device_status() == 0


@pytest.mark.parametrize("idx", [1, 2, 3, 4])
def test_planned_full_size_workloads(idx, capsys):
    """The launch configuration the benchmark times (the host work plan cuts
    requests at arbitrary tile boundaries across CTAs): the merged LSE and
    latent of every request against the oracle."""
    inp = W.make_inputs(idx, DEV)
    ns, st = mla.choose_splits(inp.spec.requests, inp.qlen, inp.heads, lengths=inp.lengths.cpu())
    plan, used = mla.plan_units(inp.lengths.cpu(), inp.qlen, inp.heads, ns)
    latent, lse_m = mla.merge(*_attend(inp, used, plan))
    torch.cuda.synchronize()
    ref = F.reference(("plain", idx), inp)
    F.check_every_row("%s with the work plan" % inp.spec.name, ref, latent, lse_m, capsys=capsys)
    assert mla.device_status() == 0


# ----------------------------------------------------------------- bad plans

def _small():
    inp_cpu = W.make_inputs(1, "cpu", lengths=[1, 17, 128, 129, 300, 1000, 0, 640])
    inp = _dev(inp_cpu)
    plan, _ = mla.plan_units(inp_cpu.lengths, inp.qlen, inp.heads, 4)
    return inp, plan


def _first_item(plan):
    G = int(plan[0])
    return 2 + G      # word index of item 0 (CTA 0's first item)


def _first_copy(plan):
    G = int(plan[0])
    return plan.numel() - 4 * G   # word index of the copy of CTA 0's first item


def _expect_flag(inp, bad):
    _attend(inp, 4, bad)
    assert mla.device_status() & mla.DEV_BAD_PLAN
    assert mla.device_status() == 0


def test_plan_for_another_grid_is_flagged():
    inp, plan = _small()
    bad = plan.clone()
    bad[0] += 1
    _expect_flag(inp, bad)


def test_plan_offsets_outside_the_buffer_are_flagged():
    inp, plan = _small()
    G = int(plan[0])
    bad = plan.clone()
    bad[1 + G] = (plan.numel() - 2 - G) // 4 - G + 1      # the last CTA's list runs past the items
    _expect_flag(inp, bad)


@pytest.mark.parametrize("field,value", [
    ("r", 8),            # request past num_requests
    ("r", -1),
    ("k", 1 | (1 << 9)),  # k >= n_r
    ("k", 0 | (5 << 9)),  # n_r > num_splits (4)
    ("k", 0 | (1 << 9) | (1 << 18)),   # row group past the groups (1)
    ("start", -128),
    ("count", 1 << 20),  # past the request's tokens
    ("count", 0),        # no tokens for a request that has some (only an empty request's one split may)
])
def test_plan_items_outside_the_launch_are_flagged(field, value):
    inp, plan = _small()
    off = {"r": 0, "k": 1, "start": 2, "count": 3}[field]
    bad = plan.clone()
    bad[_first_item(plan) + off] = value      # the item and the copy the kernel starts from
    bad[_first_copy(plan) + off] = value
    _expect_flag(inp, bad)


# ------------------------------------------------------------ prepared calls

def test_prepared_calls_match_plain_calls_and_follow_new_contents():
    """A prepared attend / merge-value call launches the same work as the
    plain call, and reads the buffers' current contents at each launch."""
    inp_cpu = W.make_inputs(1, "cpu", lengths=[1, 17, 128, 129, 300, 1000])
    inp = _dev(inp_cpu)
    plan, ns = mla.plan_units(inp_cpu.lengths, inp.qlen, inp.heads, 4)
    plan = plan.to(DEV)
    q = inp.q.clone()
    o, lse = _attend(inp, ns, plan)
    ref = mla.merge_value_gate(o, lse, inp.w_uv, inp.gate, inp.lengths, inp.qlen)
    att = mla.attend(q, inp.kv, inp.pages, inp.indptr, inp.scale, inp.kv_scale, ns, 64, heads=inp.heads,
                     plan=plan, prepare=True)
    o2, lse2 = att.outputs
    mv = mla.merge_value_gate(o2, lse2, inp.w_uv, inp.gate, inp.lengths, inp.qlen, prepare=True)
    att()
    out = mv()
    torch.cuda.synchronize()
    assert torch.equal(out, ref) and torch.equal(lse2, lse)
    # new query contents, same buffers: the prepared calls see them
    q.mul_(0.5)
    att()
    out_half = mv()
    o3, lse3 = _attend(_dev(W.Inputs(inp_cpu.spec, inp_cpu.q * 0.5, *(getattr(inp_cpu, f) for f in
                                     ("kv", "pages", "indptr", "lengths", "w_uv", "gate")),
                                     inp_cpu.scale, inp_cpu.kv_scale)), ns, plan)
    ref_half = mla.merge_value_gate(o3, lse3, inp.w_uv, inp.gate, inp.lengths, inp.qlen)
    torch.cuda.synchronize()
    assert torch.equal(out_half, ref_half) and not torch.equal(out_half, ref)
    assert mla.device_status() == 0


@pytest.mark.parametrize("heads,qlen,lengths", [
    (128, 16, [40, 3, 1]),          # 2048 rows: 43 row groups, 3 virtual CTAs of 43
    (20, 5, [150, 40, 1, 0, 700]),  # 100 rows: 3 groups of 34 (NQ 48), 50 virtual CTAs
    (1, 1, [1, 2, 300, 129]),       # a single row
])
def test_planned_row_groups_match_oracle(heads, qlen, lengths):
    """Plans for many and odd row-group counts: every group of a request runs
    the same items on its own CTA."""
    spec = W.WorkloadSpec("rows", 11, len(lengths), qlen, heads, heads + (8 if heads < 128 else 0),
                          "fixed:" + ",".join(map(str, lengths)), 0.7)
    inp_cpu = W.make_inputs(spec, "cpu", lengths=lengths)
    inp = _dev(inp_cpu)
    plan, ns = mla.plan_units(inp_cpu.lengths, qlen, heads, 3)
    o, lse = _attend(inp, ns, plan)
    _check_against_oracle(inp_cpu, o, lse, plan, ns)
    assert mla.device_status() == 0


def test_all_options_together_match_oracle():
    """fp8 query, causal mask, block tables of 16 and a work plan in one call."""
    inp_cpu = W.make_block_inputs(2, "cpu", page_size=16, lengths=[2, 3, 257, 700, 0, 129])
    inp = _dev(inp_cpu)
    q8 = (inp_cpu.q.float() * 4).to(torch.float8_e4m3fn)
    plan, ns = mla.plan_units(inp_cpu.lengths, inp.qlen, inp.heads, 4)
    o, lse = mla.attend(q8.to(DEV), inp.kv, inp.pages, inp.indptr, inp.scale, inp.kv_scale, ns, 64,
                        heads=inp.heads, qlen=inp.qlen, q_scale=0.25, causal=True, page_size=16,
                        last_page_len=inp.extra["last_page_len"], plan=plan.to(DEV))
    latent, lse_m = mla.merge(o, lse)
    torch.cuda.synchronize()
    a = dict(oracle_args(inp_cpu), q_bits=u8(q8.view(torch.uint8)), scale=inp.scale * 0.25)
    blk = _block_args(inp_cpu)
    ro, rl = O.attend_splits(**a, num_splits=ns, split_tokens=1, ranges=_plan.ranges(plan, 6, 0), causal=True,
                             q_fp8=True, **blk)
    assert_lse_close(lse, rl, "all options: partial lse")
    assert_bf16_close(o, ro, "all options: partial o", mask=np.isfinite(rl))
    rlat, rlse = O.attend(**a, causal=True, q_fp8=True, **blk)
    assert_lse_close(lse_m, rlse, "all options: merged lse")
    assert_bf16_close(latent, rlat, "all options: latent")
    assert mla.device_status() == 0


@pytest.mark.parametrize("planned", [False, True])
def test_thousands_of_short_requests(planned):
    """3,000 requests of 0-50 tokens: many 32-request windows of the unit
    cursor (round robin) or many items per CTA (plan); sampled requests and
    every empty request checked against the oracle."""
    g = torch.Generator().manual_seed(21)
    lengths = torch.randint(0, 51, (3000,), generator=g).tolist()
    spec = W.WorkloadSpec("many", 12, len(lengths), 1, 12, 12, "fixed:" + ",".join(map(str, lengths)), 0.8)
    inp_cpu = W.make_inputs(spec, "cpu", lengths=lengths)
    inp = _dev(inp_cpu)
    if planned:
        plan, ns = mla.plan_units(inp_cpu.lengths, 1, 12, 4)
        o, lse = _attend(inp, ns, plan)
    else:
        ns, st = mla.choose_splits(len(lengths), 1, 12, lengths=inp_cpu.lengths)
        o, lse = _attend(inp, ns, st=st)
    latent, lse_m = mla.merge(o, lse)
    torch.cuda.synchronize()
    lens = np.asarray(lengths)
    rng = np.random.default_rng(5)
    reqs = sorted(set(rng.choice(len(lengths), 40, replace=False).tolist()) | {int(np.argmax(lens))})
    a = dict(q_bits=bf16_bits(inp_cpu.q), kv_codes=u8(inp_cpu.kv), pages=i32(inp_cpu.pages),
             indptr=i32(inp_cpu.indptr), scale=inp.scale, kv_scale=inp.kv_scale, heads=12, qlen=1)
    rlat, rlse = O.attend(**a, requests=reqs)
    assert_lse_close(lse_m[reqs], rlse[reqs], "many requests: lse (sampled)")
    assert_bf16_close(latent[reqs], rlat[reqs], "many requests: latent (sampled)")
    empty = torch.from_numpy(lens == 0).to(DEV)
    assert torch.all(torch.isneginf(lse_m[empty])) and torch.all(latent[empty] == 0)
    assert torch.isfinite(lse_m[~empty]).all()
    assert mla.device_status() == 0
