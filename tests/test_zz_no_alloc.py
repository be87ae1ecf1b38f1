"""GPU test of mla_decode_step_static, the decode step that allocates nothing.

Some callers cannot allocate device memory while they run (a serving loop
with a fixed memory plan, a plain C host without a device allocator); this
entry point keeps the split partials in a static buffer of the library
instead.  Its results must be those of the ordinary calls with caller-owned
partials (mla_decode_attend_planned, then mla_merge_value_gate), within the
parity tolerances, on consecutive calls that reuse the buffer.

The file name sorts last so that a run stopping at its first failure has
already run every other test; the test also passes on its own in a fresh
process (it builds the library itself)."""

import pytest
import torch

import mla_decode_paged_gb300 as mla
from mla_decode_paged_gb300 import workloads as W
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
    return W.Inputs(inp.spec, *(getattr(inp, f).to(DEV) for f in
                                ("q", "kv", "pages", "indptr", "lengths", "w_uv", "gate")),
                    inp.scale, inp.kv_scale)


def _reference(inp, ns, st, plan):
    """The same step through the existing entry points, partials in torch buffers."""
    o, lse = mla.attend(inp.q, inp.kv, inp.pages, inp.indptr, inp.scale, inp.kv_scale, ns, st, heads=inp.heads,
                        qlen=inp.qlen, plan=plan)
    latent = torch.empty(o.shape[1:], dtype=torch.bfloat16, device=DEV)
    lse_m = torch.empty(lse.shape[1:], dtype=torch.float32, device=DEV)
    out = mla.merge_value_gate(o, lse, inp.w_uv, inp.gate, inp.lengths, inp.qlen, latent=latent, lse_out=lse_m)
    return out, latent, lse_m


CASES = [
    # (workload index, lengths, planned): two calls in a row with different shapes and split counts,
    # so the second reads none of what the first left in the shared buffer
    (1, [1, 17, 128, 129, 300, 1000, 0, 4000], False),
    (2, [257, 64, 700, 0, 2000], True),
    (3, [300, 129], False),
]


def test_static_step_matches_the_allocating_calls_on_consecutive_calls():
    for rep in range(2):
        for idx, lengths, planned in CASES:
            inp_cpu = W.make_inputs(idx, "cpu", lengths=lengths)
            inp = _dev(inp_cpu)
            ns, st = mla.choose_splits(len(lengths), inp.qlen, inp.heads, lengths=inp_cpu.lengths)
            plan = None
            if planned:
                plan_h, ns = mla.plan_units(inp_cpu.lengths, inp.qlen, inp.heads, ns)
                plan = plan_h.to(DEV)
            ref_out, ref_lat, ref_lse = _reference(inp, ns, st, plan)
            lse_m = torch.empty_like(ref_lse)
            out, latent, _ = mla.decode_step_static(inp.q, inp.kv, inp.pages, inp.indptr, inp.scale,
                                                    inp.kv_scale, inp.w_uv, inp.gate, inp.lengths, ns, st,
                                                    heads=inp.heads, qlen=inp.qlen, plan=plan, lse_out=lse_m)
            torch.cuda.synchronize()
            what = "call %d, workload %d" % (rep, idx)
            assert_lse_close(lse_m, to_f64(ref_lse), what + ": lse")
            assert_bf16_close(latent, to_f64(ref_lat), what + ": latent")
            assert_bf16_close(out, to_f64(ref_out), what + ": out")
            assert mla.device_status() == 0


def test_static_step_refuses_partials_above_its_buffer():
    inp = _dev(W.make_inputs(2, "cpu", lengths=[4000] * 64))
    S, H = 64 * inp.qlen, inp.heads
    ns = mla.STATIC_SCRATCH_BYTES // (S * H * 1028) + 1      # one split more than fits
    with pytest.raises(mla.MlaError, match="static") as e:
        mla.decode_step_static(inp.q, inp.kv, inp.pages, inp.indptr, inp.scale, inp.kv_scale, inp.w_uv, inp.gate,
                               inp.lengths, ns, 64, heads=H, qlen=inp.qlen)
    assert e.value.status == mla.MLA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert mla.device_status() == 0
