"""The synthetic inputs follow each workload's recipe: sizes, length
distributions, the page permutation of the pool, value distributions, the
NaN pad heads and the NaN gate rows of empty requests, and seeded
determinism.  CPU only: the large workloads are checked through their length
draws and through small-length instances of the same recipe."""

import math

import pytest
import torch

from mla_decode_paged_gb300 import workloads as W


def test_the_five_workloads():
    assert [s.name for s in W.WORKLOADS] == ["tiny_r2_h12", "decode_r64_h12", "spec_r128_q4_h12",
                                              "long_r32_h96p128", "ragged_r256_q8_h12"]
    assert [(s.requests, s.qlen, s.heads, s.heads_pad) for s in W.WORKLOADS] == [
        (2, 1, 12, 12), (64, 1, 12, 12), (128, 4, 12, 12), (32, 1, 96, 128), (256, 8, 12, 12)]
    assert [s.kv_scale for s in W.WORKLOADS] == [1.0, 0.8, 0.8, 0.8, 1.25]
    assert all(s.scale == pytest.approx(1 / math.sqrt(128 + 64)) for s in W.WORKLOADS)
    assert [s.seed for s in W.WORKLOADS] == [0, 1, 2, 3, 4]


def test_length_draws_follow_their_distributions():
    l0, l1, l2, l3, l4 = (W.draw_lengths(s) for s in W.WORKLOADS)
    assert l0.tolist() == [64, 100]
    assert l1.numel() == 64 and l1.min() >= 1024 and l1.max() <= 8192
    assert abs(l1.double().mean().item() - (1024 + 8192) / 2) < 4 * (8192 - 1024) / math.sqrt(12 * 64)
    assert l2.numel() == 128 and l2.min() >= 4096 and l2.max() <= 32768
    assert abs(l2.double().mean().item() - (4096 + 32768) / 2) < 4 * (32768 - 4096) / math.sqrt(12 * 128)
    assert l3.tolist() == [32768] * 32
    assert l4.numel() == 256 and int((l4 == 0).sum()) == 8
    nz = l4[l4 > 0].double()
    assert nz.min() >= 128 and nz.max() <= 131072
    # log-uniform: ln L is uniform on [ln 128, ln 131072] (mean 1/2, std 1/sqrt(12) once rescaled)
    u = (nz.log() - math.log(128)) / (math.log(131072) - math.log(128))
    se = 1 / math.sqrt(12 * nz.numel())
    assert abs(u.mean().item() - 0.5) < 4 * se and abs(u.std().item() - 1 / math.sqrt(12)) < 0.05
    for s in W.WORKLOADS:
        assert torch.equal(W.draw_lengths(s), W.draw_lengths(s))


def test_tiny_workload_pool_and_pages():
    """164 pages drawn without repetition from a 256-row pool."""
    inp = W.make_inputs(0)
    assert inp.kv.shape == (256, 576) and inp.pages.numel() == 164
    p = inp.pages.tolist()
    assert len(set(p)) == 164 and min(p) >= 0 and max(p) < 256
    assert inp.indptr.tolist() == [0, 64, 164] and inp.lengths.tolist() == [64, 100]


@pytest.mark.parametrize("idx", [1, 2, 3, 4])
def test_recipe_on_small_lengths(idx):
    spec = W.WORKLOADS[idx]
    lens = [0, 300, 1000, 7]
    inp = W.make_inputs(idx, lengths=lens)
    R, S, total = 4, 4 * spec.qlen, sum(lens)
    assert inp.spec.requests == R and inp.qlen == spec.qlen and inp.heads == spec.heads
    # query: bf16 N(0, 1) on the real heads, NaN on the pad heads
    assert inp.q.shape == (S, spec.heads_pad, 576) and inp.q.dtype == torch.bfloat16
    real = inp.q[:, :spec.heads].float()
    assert torch.isfinite(real).all() and abs(real.std().item() - 1) < 0.05
    if spec.heads_pad > spec.heads:
        assert torch.isnan(inp.q[:, spec.heads:].float()).all()
    # the pool holds exactly the requests' rows; the pages are a permutation of it
    assert inp.kv.shape == (total, 576) and inp.kv.dtype == torch.uint8
    assert sorted(inp.pages.tolist()) == list(range(total))
    assert inp.indptr.tolist() == [0, 0, 300, 1300, 1307]
    kv = inp.kv.view(torch.float8_e4m3fn).float()
    assert torch.isfinite(kv).all() and abs(kv.std().item() - 0.5) < 0.02
    # W_UV: bf16 N(0, 1/512); gate: bf16 N(0, 1), NaN on the rows of the empty request
    assert inp.w_uv.shape == (spec.heads, 128, 512)
    assert abs(inp.w_uv.float().std().item() - 1 / math.sqrt(512)) < 0.002
    gate = inp.gate.float().view(R, spec.qlen, spec.heads * 128)
    assert torch.isnan(gate[0]).all() and torch.isfinite(gate[1:]).all()
    assert abs(gate[1:].std().item() - 1) < 0.05
    assert inp.kv_scale == spec.kv_scale and inp.scale == spec.scale


def test_same_seed_same_inputs():
    a, b = W.make_inputs(1, lengths=[5, 600]), W.make_inputs(1, lengths=[5, 600])
    for f in ("q", "kv", "pages", "indptr", "lengths", "w_uv", "gate"):
        assert torch.equal(getattr(a, f), getattr(b, f)), f
    c = W.make_inputs(2, lengths=[5, 600])
    assert not torch.equal(a.kv, c.kv)
