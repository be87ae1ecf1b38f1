"""GPU parity of the CUDA path against the fp64 CPU oracle, element by
element, through the C ABI (via the thin binding).

Small cases span several 128-token tiles and a ragged tail; the full-size
workloads run in the launch configuration the benchmark times (split plan
from mla_choose_splits, or the host work plan) and every request of them is
checked against the oracle, whose result for each workload is computed once
per session.  Each full-size check prints its largest LSE error and its
max|err|/max|ref| to the test log."""

import math
import time

import numpy as np
import pytest
import torch

import mla_decode_paged_gb300 as mla
from mla_decode_paged_gb300 import workloads as W
from oracle import mla_oracle as O
from tests import _full as F
from tests._bits import bf16_bits, i32, oracle_args, u8
from tests.parity import assert_bf16_close, assert_lse_close

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(params=["tc", "mma"])
def kernel(request):
    """Runs a test once per attend kernel: the library's tcgen05 kernel
    (mla_decode_attend) and the warp-MMA cross-check (mla_debug_attend_mma)."""
    return request.param


def _attend(kernel, *args, **kw):
    return (mla.debug_attend_mma if kernel == "mma" else mla.attend)(*args, **kw)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mla.build()
    mla.device_status()  # clear any stale bits
    yield


def _to(inp, device):
    out = W.Inputs(inp.spec, *(getattr(inp, f).to(device) for f in
                               ("q", "kv", "pages", "indptr", "lengths", "w_uv", "gate")),
                   inp.scale, inp.kv_scale)
    return out


def _run_path(inp, ns, st, kernel="tc"):
    o, lse = _attend(kernel, inp.q, inp.kv, inp.pages, inp.indptr, inp.scale, inp.kv_scale, ns, st,
                     heads=inp.heads, qlen=inp.qlen)
    latent, lse_m = mla.merge(o, lse)
    out = mla.value_gate(latent, inp.w_uv, inp.gate, inp.lengths, inp.qlen)
    torch.cuda.synchronize()
    return o, lse, latent, lse_m, out


def _check_partials(o, lse, inp_cpu, ns, st):
    ro, rl = O.attend_splits(**oracle_args(inp_cpu), num_splits=ns, split_tokens=st)
    assert_lse_close(lse, rl, "partial lse")
    used = np.isfinite(rl)                      # o of empty / unused splits is unspecified
    assert_bf16_close(o, ro, "partial o", mask=used)


def _check_full(latent, lse_m, out, inp_cpu):
    a = oracle_args(inp_cpu)
    rlat, rlse, rout = O.decode_step(**a, w_uv_bits=bf16_bits(inp_cpu.w_uv),
                                     gate_bits=bf16_bits(inp_cpu.gate), lengths=i32(inp_cpu.lengths))
    assert_lse_close(lse_m, rlse, "merged lse")
    assert_bf16_close(latent, rlat, "latent")
    assert_bf16_close(out, rout, "out")
    empty = np.repeat(i32(inp_cpu.lengths) == 0, inp_cpu.qlen)
    if empty.any():
        assert torch.all(out[torch.from_numpy(empty).to(out.device)] == 0)


# ------------------------------------------------------------------ small cases

SMALL = [
    # (workload index, lengths)  -- spans several tiles, ragged tails, empty requests
    (0, None),
    (1, [1, 17, 128, 129, 300, 1000]),
    (2, [257, 64, 700]),
    (3, [300, 129]),
    (4, [0, 5, 200, 0, 333]),
]


@pytest.mark.parametrize("idx,lengths", SMALL)
@pytest.mark.parametrize("plan", [(1, 1 << 20), (4, 64), (8, 50), (3, 7), "auto"])
def test_small_workloads_match_oracle(idx, lengths, plan, kernel):
    inp_cpu = W.make_inputs(idx, "cpu", lengths=lengths)
    inp = _to(inp_cpu, DEV)
    if plan == "auto":
        plan = mla.choose_splits(inp.spec.requests, inp.qlen, inp.heads, lengths=inp_cpu.lengths)
    ns, st = plan
    o, lse, latent, lse_m, out = _run_path(inp, ns, st, kernel)
    _check_partials(o, lse, inp_cpu, ns, st)
    _check_full(latent, lse_m, out, inp_cpu)
    assert mla.device_status() == 0


@pytest.mark.parametrize("idx,lengths", SMALL)
def test_decode_step_matches_oracle(idx, lengths):
    """The one-call step of the public binding (split plan from max_len,
    attend, then merge + value/gate: one fused launch for these small
    batches, the two separate kernels for the 96-head one) against the
    oracle."""
    inp_cpu = W.make_inputs(idx, "cpu", lengths=lengths)
    inp = _to(inp_cpu, DEV)
    out, latent, lse_m = mla.decode_step(inp.q, inp.kv, inp.pages, inp.indptr, inp.scale, inp.kv_scale, inp.w_uv,
                                         inp.gate, inp.lengths, heads=inp.heads, qlen=inp.qlen,
                                         max_len=int(inp_cpu.lengths.max()))
    torch.cuda.synchronize()
    _check_full(latent, lse_m, out, inp_cpu)
    assert mla.device_status() == 0


@pytest.mark.parametrize("heads,qlen", [(16, 1), (12, 2), (7, 5), (16, 4), (128, 1), (20, 5), (1, 1), (128, 16)])
def test_row_counts_and_groups(heads, qlen, kernel):
    """Query-row counts that select each row-tile size and several row groups."""
    spec = W.WorkloadSpec("rows", 11, 3, qlen, heads, heads + (8 if heads < 128 else 0),
                          "fixed:150,40,1", 0.7)
    lengths = [150, 40, 1] if heads * qlen <= 512 else [40, 3, 1]
    inp_cpu = W.make_inputs(spec, "cpu", lengths=lengths)
    inp = _to(inp_cpu, DEV)
    o, lse, latent, lse_m, out = _run_path(inp, 2, 64, kernel)
    _check_partials(o, lse, inp_cpu, 2, 64)
    _check_full(latent, lse_m, out, inp_cpu)


def test_peaky_scores(kernel):
    """A large softmax scale makes attention peaky, so outputs are O(0.1-1)
    and the element-wise bound is tight."""
    inp_cpu = W.make_inputs(0, "cpu")
    inp_cpu.scale = 1.0
    inp = _to(inp_cpu, DEV)
    o, lse, latent, lse_m, out = _run_path(inp, 4, 25, kernel)
    lat_ref, _ = O.attend(**oracle_args(inp_cpu))
    assert np.abs(lat_ref).max() > 0.1
    _check_partials(o, lse, inp_cpu, 4, 25)
    _check_full(latent, lse_m, out, inp_cpu)


def test_most_splits(kernel):
    """num_splits at its cap (256): one request cut into 256 splits of 40
    tokens (the last ragged), another into 2, a third empty."""
    inp_cpu = W.make_inputs(1, "cpu", lengths=[256 * 40 - 17, 70, 0])
    inp = _to(inp_cpu, DEV)
    o, lse, latent, lse_m, out = _run_path(inp, 256, 40, kernel)
    assert torch.isfinite(lse[:, 0]).all() and torch.isfinite(lse[:2, 1]).all()
    assert torch.all(torch.isneginf(lse[2:, 1])) and torch.all(torch.isneginf(lse[:, 2]))
    _check_partials(o, lse, inp_cpu, 256, 40)
    _check_full(latent, lse_m, out, inp_cpu)
    assert mla.device_status() == 0


def test_caller_buffers_of_the_wrong_extent_are_refused():
    """Outputs the caller supplies must match the call's extent exactly:
    a smaller one would be written past its end."""
    inp = _to(W.make_inputs(0, "cpu"), DEV)
    args = (inp.q, inp.kv, inp.pages, inp.indptr, inp.scale, inp.kv_scale, 4, 25)
    small_o = torch.empty(3, 2, 12, 512, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ValueError, match="o must be"):
        mla.attend(*args, heads=12, o=small_o)
    with pytest.raises(ValueError, match="lse must be"):
        mla.attend(*args, heads=12, lse=torch.empty(4, 2, 11, device=DEV))
    o, lse = mla.attend(*args, heads=12)
    with pytest.raises(ValueError, match="latent must be"):
        mla.merge(o, lse, latent=torch.empty(2, 12, 256, dtype=torch.bfloat16, device=DEV))
    with pytest.raises(ValueError, match="out must be"):
        mla.merge_value_gate(o, lse, inp.w_uv, inp.gate, inp.lengths, out=torch.empty(2, 1000, dtype=torch.bfloat16,
                                                                                        device=DEV))
    with pytest.raises(ValueError, match="CUDA tensors|is on cpu"):
        mla.merge_value_gate(o, lse, inp.w_uv, inp.gate.cpu(), inp.lengths)
    torch.cuda.synchronize()
    assert mla.device_status() == 0


def test_all_requests_empty(kernel):
    inp_cpu = W.make_inputs(4, "cpu", lengths=[0, 0, 0])
    inp = _to(inp_cpu, DEV)
    o, lse, latent, lse_m, out = _run_path(inp, 4, 16, kernel)
    assert torch.all(torch.isneginf(lse)) and torch.all(torch.isneginf(lse_m))
    assert torch.all(latent == 0) and torch.all(out == 0)


def test_unused_splits_have_neg_inf_lse(kernel):
    inp_cpu = W.make_inputs(1, "cpu", lengths=[10, 300])
    inp = _to(inp_cpu, DEV)
    o, lse, *_ = _run_path(inp, 16, 64, kernel)
    # request 0: 1 split; request 1: ceil(300/64) = 5 splits
    assert torch.all(torch.isneginf(lse[1:, 0])) and torch.isfinite(lse[0, 0]).all()
    assert torch.isfinite(lse[:5, 1]).all() and torch.all(torch.isneginf(lse[5:, 1]))


def test_padded_heads_never_read(kernel):
    inp_cpu = W.make_inputs(3, "cpu", lengths=[70, 33])
    assert torch.isnan(inp_cpu.q[:, 96:].float()).all()
    inp = _to(inp_cpu, DEV)
    o, lse, latent, lse_m, out = _run_path(inp, 2, 40, kernel)
    assert torch.isfinite(latent).all() and torch.isfinite(out).all()
    _check_full(latent, lse_m, out, inp_cpu)


# --------------------------------------------------------------- merge / value

@pytest.mark.parametrize("splits,rows,heads", [(1, 3, 12), (5, 17, 12), (40, 9, 7), (256, 2, 3)])
def test_merge_standalone(splits, rows, heads):
    o, lse = W.make_partials(splits, rows, heads, seed=splits)
    lat, ls = mla.merge(o.to(DEV), lse.to(DEV))
    rl, rs = O.merge(O.bf16_to_f64(bf16_bits(o)), lse.double().numpy())
    assert_lse_close(ls, rs, "merge lse")
    assert_bf16_close(lat, rl, "merge latent")


@pytest.mark.parametrize("R,qlen,heads", [(3, 1, 12), (70, 1, 12), (5, 4, 12), (9, 8, 12), (2, 1, 96), (1, 3, 5),
                                          (33, 4, 12), (3, 1, 128), (40, 5, 3),
                                          # 2,000 x 12 rows: 96-row tiles on a 152-SM GB300, ragged last tile
                                          (250, 8, 12), (45, 3, 64), (1100, 1, 12)])
def test_value_gate_standalone(R, qlen, heads):
    S = R * qlen
    lat = W.make_latent(S, heads, seed=R)
    g = torch.Generator().manual_seed(R)
    w = (torch.randn(heads, 128, 512, generator=g) / math.sqrt(512)).to(torch.bfloat16)
    gate = torch.randn(S, heads * 128, generator=g).to(torch.bfloat16)
    lengths = torch.randint(0, 3, (R,), generator=g, dtype=torch.int32)
    for r in range(R):
        if lengths[r] == 0:
            gate[r * qlen:(r + 1) * qlen] = float("nan")
    out = mla.value_gate(lat.to(DEV), w.to(DEV), gate.to(DEV), lengths.to(DEV), qlen)
    ref = O.value_gate(O.bf16_to_f64(bf16_bits(lat)), bf16_bits(w), bf16_bits(gate), lengths.numpy(), qlen)
    assert_bf16_close(out, ref, "value_gate")
    dead = np.repeat(lengths.numpy() == 0, qlen)
    assert torch.all(out[torch.from_numpy(dead).to(DEV)] == 0)


def test_value_gate_tile_height_does_not_change_bytes():
    """2,000 rows x 12 heads in one call take 96-row tiles (64-row ones would
    be more than two waves of CTAs on a 152-SM GB300); the same rows as two
    calls of 1,000 take 64-row tiles.  Each row gets the same MMAs in the same
    K order and the same epilogue, so the outputs are byte-equal."""
    S, H = 2000, 12
    lat = W.make_latent(S, H, seed=9).to(DEV)
    g = torch.Generator().manual_seed(9)
    w = (torch.randn(H, 128, 512, generator=g) / math.sqrt(512)).to(torch.bfloat16).to(DEV)
    gate = torch.randn(S, H * 128, generator=g).to(torch.bfloat16).to(DEV)
    lengths = torch.randint(0, 3, (S,), generator=g, dtype=torch.int32).to(DEV)
    whole = mla.value_gate(lat, w, gate, lengths, 1)
    first = mla.value_gate(lat[:1000], w, gate[:1000], lengths[:1000], 1)
    second = mla.value_gate(lat[1000:], w, gate[1000:], lengths[1000:], 1)
    assert torch.equal(whole, torch.cat([first, second]))
    assert mla.device_status() == 0


@pytest.mark.parametrize("idx,lengths", SMALL)
def test_fused_merge_value_matches_oracle_and_two_call_path(idx, lengths):
    """mla_merge_value_gate and merge followed by value_gate, each against the
    oracle, and byte-equal to each other: both routes merge with the same row
    function and run the same 32 bf16 tensor-core MMAs (K = 16, in the same
    order) and the same sigmoid, only with 16 or 64 rows per MMA."""
    inp_cpu = W.make_inputs(idx, "cpu", lengths=lengths)
    inp = _to(inp_cpu, DEV)
    o, lse, latent, lse_m, out = _run_path(inp, 4, 40)
    lat2 = torch.empty_like(latent)
    lse2 = torch.empty_like(lse_m)
    out2 = mla.merge_value_gate(o, lse, inp.w_uv, inp.gate, inp.lengths, inp.qlen, latent=lat2, lse_out=lse2)
    torch.cuda.synchronize()
    _check_full(lat2, lse2, out2, inp_cpu)
    _check_full(latent, lse_m, out, inp_cpu)
    assert torch.equal(lat2, latent)
    assert torch.equal(torch.nan_to_num(lse2, neginf=-1e30), torch.nan_to_num(lse_m, neginf=-1e30))
    assert torch.equal(out2, out)


@pytest.mark.parametrize("splits,R,qlen,heads", [(1, 3, 1, 12), (6, 70, 1, 12), (9, 40, 8, 12), (3, 2, 1, 96),
                                                 (5, 200, 8, 12)])
def test_fused_merge_value_standalone(splits, R, qlen, heads):
    """Both routes: one launch (small batches) and merge + value (large)."""
    S = R * qlen
    o, lse = W.make_partials(splits, S, heads, seed=R)
    g = torch.Generator().manual_seed(R)
    w = (torch.randn(heads, 128, 512, generator=g) / math.sqrt(512)).to(torch.bfloat16)
    gate = torch.randn(S, heads * 128, generator=g).to(torch.bfloat16)
    lengths = torch.randint(0, 3, (R,), generator=g, dtype=torch.int32)
    out = mla.merge_value_gate(o.to(DEV), lse.to(DEV), w.to(DEV), gate.to(DEV), lengths.to(DEV), qlen)
    rl, _ = O.merge(O.bf16_to_f64(bf16_bits(o)), lse.double().numpy())
    ref = O.value_gate(rl, bf16_bits(w), bf16_bits(gate), lengths.numpy(), qlen)
    assert_bf16_close(out, ref, "fused merge+value")


# ----------------------------------------------------------------- page gather

@pytest.mark.parametrize("idx,lengths", SMALL)
def test_gather_bit_exact_small(idx, lengths):
    inp_cpu = W.make_inputs(idx, "cpu", lengths=lengths)
    inp = _to(inp_cpu, DEV)
    rows = mla.debug_gather(inp.kv, inp.pages, inp.indptr)
    ref = O.gather_all(u8(inp_cpu.kv), i32(inp_cpu.pages), i32(inp_cpu.indptr))
    assert np.array_equal(u8(rows), ref)


def test_gather_bit_exact_full_decode_batch():
    inp = W.make_inputs(1, DEV)
    rows = mla.debug_gather(inp.kv, inp.pages, inp.indptr)
    ref = O.gather_all(u8(inp.kv), i32(inp.pages), i32(inp.indptr))
    assert np.array_equal(u8(rows), ref)


def test_bad_pages_and_indptr_are_flagged_not_faulted(kernel):
    inp_cpu = W.make_inputs(0, "cpu")
    inp = _to(inp_cpu, DEV)
    bad = inp.pages.clone()
    bad[3] = inp.kv.shape[0] + 5          # outside the pool: clamped + flagged
    bad[7] = -2
    _attend(kernel, inp.q, inp.kv, bad, inp.indptr, inp.scale, inp.kv_scale, 1, 1 << 20)
    assert mla.device_status() & mla.DEV_BAD_PAGE
    bad_ip = inp.indptr.clone()
    bad_ip[1] = bad_ip[2] + 1             # decreasing: request treated as empty + flagged
    _attend(kernel, inp.q, inp.kv, inp.pages, bad_ip, inp.scale, inp.kv_scale, 1, 1 << 20)
    assert mla.device_status() & mla.DEV_BAD_INDPTR
    assert mla.device_status() == 0


def test_a_wait_that_runs_out_is_reported_and_the_context_survives():
    """A kernel waits, through the bounded wait every kernel here uses, on a
    barrier nothing completes: it gives up after its budget (~2 s), flags
    DEV_TIMEOUT and exits; the next step on the same context is exact."""
    assert mla.device_status() == 0
    t0 = time.time()
    mla.debug_wait_timeout()
    assert mla.device_status() & mla.DEV_TIMEOUT
    assert time.time() - t0 < 60
    inp_cpu = W.make_inputs(0, "cpu")
    inp = _to(inp_cpu, DEV)
    o, lse, latent, lse_m, out = _run_path(inp, 4, 25)
    _check_full(latent, lse_m, out, inp_cpu)
    assert mla.device_status() == 0


# ------------------------------------------------------------ full-size workloads

@pytest.mark.parametrize("idx", [1, 2, 3, 4])
def test_full_size_workloads_every_request(idx, kernel, capsys):
    """The benchmark's workloads at full size, launched with the split plan
    of mla_choose_splits: merged LSE, latent and output of every request
    against the oracle (computed once per workload and shared)."""
    inp = W.make_inputs(idx, DEV)
    ns, st = mla.choose_splits(inp.spec.requests, inp.qlen, inp.heads, lengths=inp.lengths.cpu())
    _, _, latent, lse_m, out = _run_path(inp, ns, st, kernel)
    ref = F.reference(("plain", idx), inp)
    F.check_every_row("%s (%s kernel)" % (inp.spec.name, kernel), ref, latent, lse_m, out, capsys)
    lens = i32(inp.lengths)
    dead = torch.from_numpy(np.repeat(lens == 0, inp.qlen)).to(DEV)
    assert torch.all(out[dead] == 0) and torch.all(torch.isneginf(lse_m[dead]))
    assert mla.device_status() == 0


@pytest.mark.parametrize("idx,ns,st,lo,hi", [(2, 32, 512, 8, 32), (3, 16, 2048, 16, 16)])
def test_workloads_at_their_stated_split_counts(idx, ns, st, lo, hi, kernel, capsys):
    """Workloads cut the way their descriptions state, under the split rule:
    the speculative-decode one into 8 to 32 split-KV partials per request
    (32 splits of 512 tokens), the 96-head long-context one into 16 (heavy
    split-KV: 16 splits of 2,048 tokens); then the LSE merge and W_UV + gate.
    Merged results of every request against the oracle (the same reference
    as any other cut); the partials of sampled requests against the oracle's
    per-split attention."""
    inp = W.make_inputs(idx, DEV)
    lens = i32(inp.lengths)
    n_r = np.minimum(ns, np.maximum(1, -(-lens // st)))
    assert n_r.min() >= lo and n_r.max() <= hi
    o, lse, latent, lse_m, out = _run_path(inp, ns, st, kernel)
    ref = F.reference(("plain", idx), inp)
    F.check_every_row("%s, %d-%d partials (%s kernel)" % (inp.spec.name, n_r.min(), n_r.max(), kernel), ref, latent,
                      lse_m, out, capsys)
    inp_cpu = _to(inp, "cpu")   # the same bytes (a CPU generator would draw others)
    reqs = sorted({int(np.argmin(lens)), int(np.argmax(lens)), 17, len(lens) - 1})
    ro, rl = O.attend_splits(**oracle_args(inp_cpu), num_splits=ns, split_tokens=st, requests=reqs)
    rows = np.concatenate([np.arange(r * inp.qlen, (r + 1) * inp.qlen) for r in reqs])
    sel = torch.from_numpy(rows).to(DEV)
    assert_lse_close(lse[:, sel], rl[:, rows], "partial lse (stated split count)")
    assert_bf16_close(o[:, sel], ro[:, rows], "partial o (stated split count)", mask=np.isfinite(rl[:, rows]))
    assert mla.device_status() == 0


# ------------------------------------------------------------- causal option

CAUSAL_SMALL = [
    # (workload index, lengths): qlen 4 / 8, requests shorter than qlen, several tiles, a ragged tail
    (2, [2, 3, 257, 700]),
    (4, [0, 5, 7, 200, 333]),
    (2, [130, 1, 4]),
]


@pytest.mark.parametrize("idx,lengths", CAUSAL_SMALL)
@pytest.mark.parametrize("plan", [(1, 1 << 20), (4, 64), (8, 50), (3, 7)])
def test_causal_small_workloads_match_oracle(idx, lengths, plan):
    inp_cpu = W.make_inputs(idx, "cpu", lengths=lengths)
    inp = _to(inp_cpu, DEV)
    ns, st = plan
    o, lse = mla.attend(inp.q, inp.kv, inp.pages, inp.indptr, inp.scale, inp.kv_scale, ns, st,
                        heads=inp.heads, qlen=inp.qlen, causal=True)
    latent, lse_m = mla.merge(o, lse)
    out = mla.value_gate(latent, inp.w_uv, inp.gate, inp.lengths, inp.qlen)
    torch.cuda.synchronize()
    a = oracle_args(inp_cpu)
    ro, rl = O.attend_splits(**a, num_splits=ns, split_tokens=st, causal=True)
    assert_lse_close(lse, rl, "causal partial lse")
    assert_bf16_close(o, ro, "causal partial o", mask=np.isfinite(rl))
    # a split a row sees nothing of: o written as 0, not left unspecified
    seen_none = np.isneginf(rl) & ~np.isnan(ro[..., 0])
    if seen_none.any():
        assert torch.all(o[torch.from_numpy(seen_none).to(DEV)] == 0)
    rlat, rlse, rout = O.decode_step(**a, w_uv_bits=bf16_bits(inp_cpu.w_uv), gate_bits=bf16_bits(inp_cpu.gate),
                                     lengths=i32(inp_cpu.lengths), causal=True)
    assert_lse_close(lse_m, rlse, "causal merged lse")
    assert_bf16_close(latent, rlat, "causal latent")
    assert_bf16_close(out, rout, "causal out")
    assert mla.device_status() == 0


def test_causal_is_exactly_unmasked_at_qlen_1():
    inp = _to(W.make_inputs(1, "cpu", lengths=[1, 17, 128, 129, 300]), DEV)
    a = mla.attend(inp.q, inp.kv, inp.pages, inp.indptr, inp.scale, inp.kv_scale, 4, 64, heads=inp.heads)
    b = mla.attend(inp.q, inp.kv, inp.pages, inp.indptr, inp.scale, inp.kv_scale, 4, 64, heads=inp.heads,
                   causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1])
    used = torch.isfinite(a[1])                 # o of unused splits is unspecified
    assert torch.equal(a[0][used], b[0][used])


@pytest.mark.parametrize("idx", [2, 4])
def test_causal_full_size_every_request(idx, capsys):
    inp = W.make_inputs(idx, DEV)
    ns, st = mla.choose_splits(inp.spec.requests, inp.qlen, inp.heads, lengths=inp.lengths.cpu())
    out, latent, lse_m = mla.decode_step(inp.q, inp.kv, inp.pages, inp.indptr, inp.scale, inp.kv_scale, inp.w_uv,
                                         inp.gate, inp.lengths, heads=inp.heads, qlen=inp.qlen, num_splits=ns,
                                         split_tokens=st, causal=True)
    torch.cuda.synchronize()
    ref = F.reference(("causal", idx), inp, causal=True)
    F.check_every_row("%s causal" % inp.spec.name, ref, latent, lse_m, out, capsys)
    assert mla.device_status() == 0


# ------------------------------------------------------- block-table caches

def _to_blocks(inp, device):
    out = _to(inp, device)
    out.extra["page_size"] = inp.extra["page_size"]
    out.extra["last_page_len"] = inp.extra["last_page_len"].to(device)
    return out


@pytest.mark.parametrize("P,idx,lengths", [(2, 4, [0, 5, 200, 0, 333]), (16, 1, [1, 17, 128, 129, 300, 1000]),
                                           (64, 2, [257, 64, 700]), (16, 3, [300, 129]),
                                           (128, 4, [0, 129, 640]),             # a block per tile
                                           (256, 1, [1, 300, 1000, 256])])      # largest block: tiles share one
@pytest.mark.parametrize("plan", [(1, 1 << 20), (4, 64), (3, 7)])
def test_block_table_small_workloads_match_oracle(P, idx, lengths, plan):
    inp_cpu = W.make_block_inputs(idx, "cpu", page_size=P, lengths=lengths)
    inp = _to_blocks(inp_cpu, DEV)
    last = inp.extra["last_page_len"]
    ns, st = plan
    o, lse = mla.attend(inp.q, inp.kv, inp.pages, inp.indptr, inp.scale, inp.kv_scale, ns, st, heads=inp.heads,
                        qlen=inp.qlen, page_size=P, last_page_len=last)
    latent, lse_m = mla.merge(o, lse)
    torch.cuda.synchronize()
    a = oracle_args(inp_cpu)
    lp = i32(inp_cpu.extra["last_page_len"])
    ro, rl = O.attend_splits(**a, num_splits=ns, split_tokens=st, page_size=P, last_page_len=lp)
    assert_lse_close(lse, rl, "block-table partial lse")
    assert_bf16_close(o, ro, "block-table partial o", mask=np.isfinite(rl))
    rlat, rlse = O.attend(**a, page_size=P, last_page_len=lp)
    assert_lse_close(lse_m, rlse, "block-table merged lse")
    assert_bf16_close(latent, rlat, "block-table latent")
    assert mla.device_status() == 0


def test_block_table_causal_matches_oracle():
    inp_cpu = W.make_block_inputs(2, "cpu", page_size=16, lengths=[2, 3, 257, 700])
    inp = _to_blocks(inp_cpu, DEV)
    o, lse = mla.attend(inp.q, inp.kv, inp.pages, inp.indptr, inp.scale, inp.kv_scale, 4, 64, heads=inp.heads,
                        qlen=inp.qlen, page_size=16, last_page_len=inp.extra["last_page_len"], causal=True)
    latent, lse_m = mla.merge(o, lse)
    torch.cuda.synchronize()
    rlat, rlse = O.attend(**oracle_args(inp_cpu), page_size=16, last_page_len=i32(inp_cpu.extra["last_page_len"]),
                          causal=True)
    assert_lse_close(lse_m, rlse, "block-table causal lse")
    assert_bf16_close(latent, rlat, "block-table causal latent")
    assert mla.device_status() == 0


def test_block_table_full_decode_batch_every_request(capsys):
    inp = W.make_block_inputs(1, DEV, page_size=16)
    ns, st = mla.choose_splits(inp.spec.requests, inp.qlen, inp.heads, lengths=inp.lengths.cpu())
    last = inp.extra["last_page_len"]
    o, lse = mla.attend(inp.q, inp.kv, inp.pages, inp.indptr, inp.scale, inp.kv_scale, ns, st, heads=inp.heads,
                        page_size=16, last_page_len=last)
    latent, lse_m = mla.merge(o, lse)
    torch.cuda.synchronize()
    ref = F.reference(("blocks16", 1), inp, page_size=16, last_page_len=last, with_out=False)
    F.check_every_row("decode_r64_h12, block tables of 16", ref, latent, lse_m, capsys=capsys)
    assert mla.device_status() == 0


def test_block_table_bad_last_page_len_is_flagged_not_faulted():
    inp = _to_blocks(W.make_block_inputs(1, "cpu", page_size=16, lengths=[40, 300]), DEV)
    last = inp.extra["last_page_len"].clone()
    last[1] = 17                                         # more rows than a block holds
    mla.attend(inp.q, inp.kv, inp.pages, inp.indptr, inp.scale, inp.kv_scale, 2, 64, heads=inp.heads,
               page_size=16, last_page_len=last)
    assert mla.device_status() & mla.DEV_BAD_INDPTR
    assert mla.device_status() == 0


@pytest.mark.parametrize("ranks", [2, 4])
def test_second_level_combine_of_sharded_partials(ranks):
    """Partials computed separately over each decode-context-parallel shard
    (token i of a request on rank i % ranks), concatenated along the split
    axis and merged by mla_merge_splits: the full attention."""
    from tests.test_oracle import _shard_by_slot
    inp_cpu = W.make_inputs(4, "cpu", lengths=[0, 5, 200, 333, 1, 700])
    inp = _to(inp_cpu, DEV)
    a = oracle_args(inp_cpu)
    os_, ls_ = [], []
    for k, (pg, ip) in enumerate(_shard_by_slot(a["pages"], a["indptr"], ranks)):
        o, lse = mla.attend(inp.q, inp.kv, torch.from_numpy(pg).to(DEV), torch.from_numpy(ip).to(DEV), inp.scale,
                            inp.kv_scale, 2 + k, 64, heads=inp.heads, qlen=inp.qlen)
        os_.append(o)
        ls_.append(lse)
    latent, lse_m = mla.merge(torch.cat(os_).contiguous(), torch.cat(ls_).contiguous())
    torch.cuda.synchronize()
    rlat, rlse = O.attend(**a)
    assert_lse_close(lse_m, rlse, "combined lse")
    assert_bf16_close(latent, rlat, "combined latent")
    assert mla.device_status() == 0


# ------------------------------------------------------------ fp8 query

def _q8(inp_cpu, gain=4.0):
    """An fp8 query of the workload's shape (codes from q * gain, NaN pad heads kept)."""
    return (inp_cpu.q.float() * gain).to(torch.float8_e4m3fn)


@pytest.mark.parametrize("idx,lengths", [(1, [1, 17, 128, 129, 300, 1000]), (2, [257, 64, 700]), (3, [300, 129]),
                                         (4, [0, 5, 200, 0, 333])])
@pytest.mark.parametrize("plan", [(1, 1 << 20), (4, 64), (3, 7)])
def test_fp8_query_small_workloads_match_oracle(idx, lengths, plan):
    inp_cpu = W.make_inputs(idx, "cpu", lengths=lengths)
    inp = _to(inp_cpu, DEV)
    q8 = _q8(inp_cpu)
    q_scale = 0.25
    ns, st = plan
    o, lse = mla.attend(q8.to(DEV), inp.kv, inp.pages, inp.indptr, inp.scale, inp.kv_scale, ns, st,
                        heads=inp.heads, qlen=inp.qlen, q_scale=q_scale)
    latent, lse_m = mla.merge(o, lse)
    torch.cuda.synchronize()
    a = dict(oracle_args(inp_cpu), q_bits=u8(q8.view(torch.uint8)), scale=inp.scale * q_scale)
    ro, rl = O.attend_splits(**a, num_splits=ns, split_tokens=st, q_fp8=True)
    assert_lse_close(lse, rl, "fp8-q partial lse")
    assert_bf16_close(o, ro, "fp8-q partial o", mask=np.isfinite(rl))
    rlat, rlse = O.attend(**a, q_fp8=True)
    assert_lse_close(lse_m, rlse, "fp8-q merged lse")
    assert_bf16_close(latent, rlat, "fp8-q latent")
    assert mla.device_status() == 0


def test_fp8_query_full_size_every_request(capsys):
    inp = W.make_inputs(2, DEV)
    q8 = (inp.q.float() * 4).to(torch.float8_e4m3fn)
    ns, st = mla.choose_splits(inp.spec.requests, inp.qlen, inp.heads, lengths=inp.lengths.cpu())
    o, lse = mla.attend(q8, inp.kv, inp.pages, inp.indptr, inp.scale, inp.kv_scale, ns, st, heads=inp.heads,
                        qlen=inp.qlen, q_scale=0.25)
    latent, lse_m = mla.merge(o, lse)
    torch.cuda.synchronize()
    ref = F.reference(("q8", 2), inp, q_codes=q8.view(torch.uint8), q_scale=0.25, with_out=False)
    F.check_every_row("spec_r128_q4_h12, fp8 query", ref, latent, lse_m, capsys=capsys)
    assert mla.device_status() == 0


# ------------------------------------------- rising scores (reference moves)

def _rising_keys(inp_cpu, gain=100.0):
    """The workload's KV rows with their 64 rope values (key only: the value
    is the 512 latent values) scaled by 1 + (gain - 1) * pos / L inside each
    request (page size 1), so each 128-token tile's largest score lies far
    above every earlier tile's: the kernel's lazy reference max moves, and the
    O accumulated so far is rescaled, on most tiles of a unit, while the
    values keep their ordinary size."""
    kv = inp_cpu.kv.view(torch.float8_e4m3fn).float()
    pages, indptr = inp_cpu.pages.long(), inp_cpu.indptr.long()
    for r in range(len(indptr) - 1):
        rows = pages[indptr[r]:indptr[r + 1]]
        n = len(rows)
        if n:
            g = 1.0 + (gain - 1.0) * torch.arange(n, dtype=torch.float32) / max(n - 1, 1)
            kv[rows, 512:] *= g[:, None]
    inp_cpu.kv = kv.to(torch.float8_e4m3fn).view(torch.uint8)
    return inp_cpu


@pytest.mark.parametrize("idx,lengths", [(1, [1, 200, 1000, 2000]), (2, [700, 1500]), (4, [0, 300, 1200])])
@pytest.mark.parametrize("mode", ["split rule", "plan", "causal"])
def test_rising_scores_move_the_reference_and_match_oracle(idx, lengths, mode, kernel, capsys):
    if kernel == "mma" and mode != "split rule":
        pytest.skip("the warp-MMA cross-check kernel takes no work plan and no mask")
    inp_cpu = _rising_keys(W.make_inputs(idx, "cpu", lengths=lengths))
    inp = _to(inp_cpu, DEV)
    ns, st, kw = 3, 512, {}
    if mode == "plan":
        plan_h, ns = mla.plan_units(inp_cpu.lengths, inp.qlen, inp.heads, 4)
        kw["plan"] = plan_h.to(DEV)
    if mode == "causal":
        kw["causal"] = True
    o, lse = _attend(kernel, inp.q, inp.kv, inp.pages, inp.indptr, inp.scale, inp.kv_scale, ns, st,
                     heads=inp.heads, qlen=inp.qlen, **kw)
    latent, lse_m = mla.merge(o, lse)
    out = mla.value_gate(latent, inp.w_uv, inp.gate, inp.lengths, inp.qlen)
    torch.cuda.synchronize()
    a = oracle_args(inp_cpu)
    rlat, rlse, rout = O.decode_step(**a, w_uv_bits=bf16_bits(inp_cpu.w_uv), gate_bits=bf16_bits(inp_cpu.gate),
                                     lengths=i32(inp_cpu.lengths), causal=mode == "causal")
    assert np.nanmax(np.abs(rlse[np.isfinite(rlse)])) > 20      # scores far beyond the first tile's
    F.check_every_row("%s rising scores (%s, %s)" % (inp.spec.name, kernel, mode), (rlat, rlse, rout), latent,
                      lse_m, out, capsys)
    assert mla.device_status() == 0


# ------------------------------------------------------ outlier-channel query

def _outlier_query(inp_cpu, rope_gain=64.0, chan_gain=100.0, chans=(7, 100, 300)):
    """The workload's query with outlier channels: the 64 rope dims scaled by
    rope_gain and a few latent channels by chan_gain in every row, so that a
    row's largest element is far above most of it (the per-row scale of the
    two-term e4m3 query then leaves the ordinary elements small)."""
    q = inp_cpu.q.float()
    q[..., 512:] *= rope_gain
    q[..., list(chans)] *= chan_gain
    inp_cpu.q = q.to(torch.bfloat16)
    return inp_cpu


@pytest.mark.parametrize("idx,lengths", [(1, [1, 17, 128, 129, 300, 1000]), (2, [257, 64, 700]),
                                         (3, [300, 129]), (4, [0, 5, 200, 0, 333])])
@pytest.mark.parametrize("planned", [False, True])
def test_outlier_channel_query_matches_oracle(idx, lengths, planned, kernel, capsys):
    if planned and kernel == "mma":
        pytest.skip("the warp-MMA cross-check kernel takes no work plan")
    inp_cpu = _outlier_query(W.make_inputs(idx, "cpu", lengths=lengths))
    inp = _to(inp_cpu, DEV)
    ns, st = 3, 128
    plan = None
    if planned:
        plan_h, ns = mla.plan_units(inp_cpu.lengths, inp.qlen, inp.heads, 4)
        plan = plan_h.to(DEV)
    kw = {} if plan is None else {"plan": plan}
    o, lse = _attend(kernel, inp.q, inp.kv, inp.pages, inp.indptr, inp.scale, inp.kv_scale, ns, st,
                     heads=inp.heads, qlen=inp.qlen, **kw)
    latent, lse_m = mla.merge(o, lse)
    out = mla.value_gate(latent, inp.w_uv, inp.gate, inp.lengths, inp.qlen)
    torch.cuda.synchronize()
    a = oracle_args(inp_cpu)
    rlat, rlse, rout = O.decode_step(**a, w_uv_bits=bf16_bits(inp_cpu.w_uv), gate_bits=bf16_bits(inp_cpu.gate),
                                     lengths=i32(inp_cpu.lengths))
    assert np.nanmax(np.abs(rlse[np.isfinite(rlse)])) > 10      # the outliers dominate the scores
    F.check_every_row("%s outlier-channel query (%s, %s)" % (inp.spec.name, kernel, "plan" if planned else "split rule"),
                      (rlat, rlse, rout), latent, lse_m, out, capsys)
    assert mla.device_status() == 0
