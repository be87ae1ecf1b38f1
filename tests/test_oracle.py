"""CPU pins of the oracle: each test ties it to something other than itself
(closed forms, the OCP FP8 table, library routines, invariants of softmax
attention, and an independent scalar brute force)."""

import math
import os

import numpy as np
import pytest
import torch

from mla_decode_paged_gb300 import workloads as W
from oracle import brute, mla_oracle as O
from tests._bits import bf16_bits, oracle_args, u8, i32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


# --------------------------------------------------------------------- formats

def test_e4m3_all_codes_match_torch_cast():
    codes = np.arange(256, dtype=np.uint8)
    ours = O.e4m3fn_to_f64(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.array_equal(np.signbit(ours[ok]), np.signbit(ref[ok]))
    # the brute force's decoder agrees code by code
    b = np.array([brute.fp8_e4m3fn(int(c)) for c in codes])
    assert np.array_equal(np.isnan(b), np.isnan(ref)) and np.array_equal(b[ok], ref[ok])


def test_e4m3_ocp_table_values():
    for code, val in _golden_rows("e4m3fn_ocp.txt"):
        c = int(code, 16)
        got = float(O.e4m3fn_to_f64(np.array([c], np.uint8))[0])
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def test_bf16_decode_matches_torch():
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(4096, generator=g) * 100).to(torch.bfloat16)
    x[:4] = torch.tensor([0.0, -0.0, float("inf"), float("nan")])
    ours = O.bf16_to_f64(bf16_bits(x))
    ref = x.to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])


def test_sigmoid_special_points():
    assert O.sigmoid(0.0) == 0.5
    assert O.sigmoid(np.inf) == 1.0 and O.sigmoid(-np.inf) == 0.0
    x = np.linspace(-20, 20, 81)
    assert np.allclose(O.sigmoid(x) + O.sigmoid(-x), 1.0, atol=1e-15)
    assert np.allclose(O.sigmoid(x), 0.5 * (1 + np.tanh(x / 2)), atol=1e-15)


# ------------------------------------------------------------------ split plan

def test_split_plan_golden():
    for L, ns, st, *ranges in _golden_rows("split_plan.txt"):
        want = [tuple(int(v) for v in r.split(":")) for r in ranges]
        assert O.split_plan(int(L), int(ns), int(st)) == want, (L, ns, st)


@pytest.mark.parametrize("L", [0, 1, 2, 31, 64, 1000, 4097])
@pytest.mark.parametrize("ns,st", [(1, 64), (4, 16), (32, 128), (7, 3)])
def test_split_plan_partitions(L, ns, st):
    plan = O.split_plan(L, ns, st)
    assert 1 <= len(plan) <= ns
    assert plan[0][0] == 0 and plan[-1][1] == L
    for (a, b), (c, d) in zip(plan, plan[1:]):
        assert b == c
    lens = [b - a for a, b in plan]
    assert max(lens) - min(lens) <= 1
    assert len(plan) == max(1, min(ns, -(-L // st)))


# --------------------------------------------------------------- closed forms

def _tiny_case():
    kv = np.zeros((4, 576), np.uint8)
    kv[2, 0], kv[2, 1] = 0x38, 0x30   # token 0 (page 2): 1.0, 0.5
    kv[0, 0], kv[0, 1] = 0x40, 0xB8   # token 1 (page 0): 2.0, -1.0
    q = np.zeros((1, 1, 576), np.uint16)
    q[0, 0, 0] = 0x3F80               # 1.0
    pages = np.array([2, 0], np.int32)
    indptr = np.array([0, 2], np.int32)
    return q, kv, pages, indptr


def test_tiny_closed_form_golden():
    g = {k: float(v) for k, v in _golden_rows("tiny_closed_form.txt")}
    q, kv, pages, indptr = _tiny_case()
    lat, lse, ps = O.attend(q, kv, pages, indptr, 1.0, 1.0, 1, 1, return_p=True)
    assert abs(lse[0, 0] - g["lse"]) < 1e-14
    assert np.allclose(ps[0][0, 0], [g["p0"], g["p1"]], atol=1e-15, rtol=0)
    assert abs(lat[0, 0, 0] - g["latent0"]) < 1e-14
    assert abs(lat[0, 0, 1] - g["latent1"]) < 1e-14
    assert np.all(lat[0, 0, 2:] == 0)


def test_one_token_context_returns_that_row():
    rng = np.random.default_rng(5)
    kv = rng.integers(0, 256, (8, 576), dtype=np.uint8)
    kv[(kv & 0x7F) == 0x7F] = 0x11          # no NaN codes
    q = bf16_bits(torch.randn(3, 4, 576, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16))
    pages = np.array([5, 1, 7], np.int32)
    indptr = np.array([0, 1, 2, 3], np.int32)
    lat, lse = O.attend(q, kv, pages, indptr, 0.3, 1.5, 4, 1)
    for r, page in enumerate(pages):
        row = np.array([brute.fp8_e4m3fn(int(c)) * 1.5 for c in kv[page]])
        for h in range(4):
            assert np.array_equal(lat[r, h], row[:512])            # p = 1 exactly
            qv = np.array([brute.bf16(int(b)) for b in q[r, h]])
            assert abs(lse[r, h] - 0.3 * math.fsum(qv * row)) < 1e-12


def test_softmax_weights_sum_to_one():
    inp = W.make_inputs(0)
    lat, lse, ps = O.attend(**oracle_args(inp), return_p=True)
    for r, p in ps.items():
        assert p.shape[-1] == [64, 100][r]
        assert np.allclose(p.sum(-1), 1.0, atol=1e-13)
        assert np.all(p >= 0)


def test_constant_value_rows_give_that_row():
    row = (np.arange(576) * 37 % 120).astype(np.uint8)
    kv = np.tile(row, (10, 1))
    q = bf16_bits(torch.randn(1, 3, 576, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16))
    pages = np.array([9, 3, 4, 0, 7], np.int32)
    lat, _ = O.attend(q, kv, pages, np.array([0, 5], np.int32), 0.1, 0.8, 3, 1)
    want = O.e4m3fn_to_f64(row)[:512] * 0.8
    assert np.allclose(lat[0], want[None, :], atol=1e-14, rtol=1e-14)


def test_zero_query_gives_mean_of_values():
    inp = W.make_inputs(0)
    args = oracle_args(inp)
    args["q_bits"] = np.zeros_like(args["q_bits"])
    lat, lse = O.attend(**args)
    for r in range(2):
        rows = O.gather_rows(args["kv_codes"], args["pages"], args["indptr"], r)
        vals = rows.view(np.uint8)
        mean = torch.from_numpy(vals.copy()).view(torch.float8_e4m3fn).to(torch.float64).mean(0).numpy()
        assert np.allclose(lat[r], mean[None, :512] * inp.kv_scale, atol=1e-14)
        assert np.allclose(lse[r], math.log(rows.shape[0]), atol=1e-14)


def test_empty_request_zero_even_with_nan_gate():
    inp = W.make_inputs(0, lengths=[0, 5])
    a = oracle_args(inp)
    gate = bf16_bits(inp.gate)
    assert np.isnan(O.bf16_to_f64(gate[0])).all()
    lat, lse, out = O.decode_step(**a, w_uv_bits=bf16_bits(inp.w_uv), gate_bits=gate,
                                  lengths=i32(inp.lengths))
    assert np.all(lat[0] == 0) and np.all(lse[0] == -np.inf)
    assert np.all(out[0] == 0) and np.isfinite(out[1]).all()


def test_padded_heads_are_ignored():
    inp = W.make_inputs(3, lengths=[3, 2])
    a = oracle_args(inp)
    assert np.isnan(O.bf16_to_f64(a["q_bits"][:, 96:])).all()
    lat, lse = O.attend(**a)
    assert np.isfinite(lat).all() and np.isfinite(lse).all()
    a2 = dict(a)
    a2["q_bits"] = np.ascontiguousarray(a["q_bits"][:, :96])
    lat2, lse2 = O.attend(**a2)
    assert np.array_equal(lat, lat2) and np.array_equal(lse, lse2)


# ------------------------------------------------------------- split + merge

@pytest.mark.parametrize("ns,st", [(1, 1 << 20), (4, 16), (4, 25), (7, 9), (64, 1)])
def test_merge_of_splits_equals_unsplit(ns, st):
    inp = W.make_inputs(0)
    a = oracle_args(inp)
    lat, lse = O.attend(**a)
    o, ls = O.attend_splits(**a, num_splits=ns, split_tokens=st)
    mlat, mlse = O.merge(o, ls)
    assert np.allclose(mlat, lat, atol=1e-12, rtol=1e-12)
    assert np.allclose(mlse, lse, atol=1e-12, rtol=0)


def test_merge_of_random_partition_equals_unsplit():
    inp = W.make_inputs(0)
    a = oracle_args(inp)
    lat, lse = O.attend(**a)
    rng = np.random.default_rng(11)
    for r in range(2):
        K = O.dequant(O.gather_rows(a["kv_codes"], a["pages"], a["indptr"], r), inp.kv_scale)
        rows = O.bf16_to_f64(a["q_bits"][r, :12])
        cuts = np.sort(rng.choice(np.arange(1, K.shape[0]), size=6, replace=False))
        edges = [0, *cuts.tolist(), K.shape[0]]
        os_, ls_ = [], []
        for x, y in zip(edges, edges[1:]):
            l_, s_, _ = O.attend_rows(rows, K[x:y], inp.scale)
            os_.append(l_[None])
            ls_.append(s_[None])
        ml, ms = O.merge(np.concatenate(os_)[:, None], np.concatenate(ls_)[:, None])
        assert np.allclose(ml[0], lat[r], atol=1e-12)
        assert np.allclose(ms[0], lse[r], atol=1e-12)


def _random_ranges(lengths, num_splits, rng):
    """A random partition of each request's tokens into 1..num_splits
    consecutive ranges (some possibly empty)."""
    out = []
    for L in lengths:
        n = int(rng.integers(1, num_splits + 1))
        cuts = np.sort(rng.integers(0, L + 1, size=n - 1)) if L > 0 else np.zeros(n - 1, dtype=int)
        edges = [0, *cuts.tolist(), int(L)]
        out.append(list(zip(edges, edges[1:])))
    return out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_merge_over_explicit_ranges_equals_unsplit(seed):
    """Any partition of the tokens, merged by LSE, gives the unsplit
    attention: the identity every split layout rests on."""
    inp = W.make_inputs(1, lengths=[0, 1, 17, 128, 129, 300])
    a = oracle_args(inp)
    lat, lse = O.attend(**a)
    rng = np.random.default_rng(seed)
    rg = _random_ranges(i32(inp.lengths), 5, rng)
    o, ls = O.attend_splits(**a, num_splits=5, split_tokens=1, ranges=rg)
    for r, cuts in enumerate(rg):           # splits past a request's ranges stay unused
        assert np.all(np.isneginf(ls[len(cuts):, r]))
        for k, (x, y) in enumerate(cuts):
            assert (x == y) == bool(np.all(np.isneginf(ls[k, r])))
    mlat, mlse = O.merge(o, ls)
    assert np.allclose(mlat, lat, atol=1e-12, rtol=1e-12)
    assert np.array_equal(np.isneginf(mlse), np.isneginf(lse))
    f = np.isfinite(lse)
    assert np.allclose(mlse[f], lse[f], atol=1e-12)


def test_explicit_ranges_causal_merge_equals_unsplit():
    a, _, _, _ = _spec_like(seed=3)
    lens = [int(a["indptr"][r + 1] - a["indptr"][r]) for r in range(len(a["indptr"]) - 1)]
    rg = _random_ranges(lens, 4, np.random.default_rng(9))
    lat, lse = O.attend(**a, causal=True)
    o, ls = O.attend_splits(**a, num_splits=4, split_tokens=1, causal=True, ranges=rg)
    mlat, mlse = O.merge(o, ls)
    assert np.allclose(mlat, lat, atol=1e-12, rtol=1e-12)
    assert np.array_equal(np.isneginf(mlse), np.isneginf(lse))
    f = np.isfinite(lse)
    assert np.allclose(mlse[f], lse[f], atol=1e-12)


def test_merge_matches_brute_and_skips_empty():
    o_t, lse_t = W.make_partials(5, 4, 3, seed=1)
    o = O.bf16_to_f64(bf16_bits(o_t))[..., :8]
    lse = lse_t.to(torch.float64).numpy()
    lat, ls = O.merge(o, lse)
    blat, bls = brute.merge(o.tolist(), lse.tolist())
    assert np.allclose(lat, np.array(blat), atol=1e-12)
    assert np.array_equal(np.isinf(ls), np.isinf(np.array(bls)))
    fin = np.isfinite(ls)
    assert np.allclose(ls[fin], np.array(bls)[fin], atol=1e-12)
    assert np.all(lat[2] == 0) and np.all(np.isneginf(ls[2]))    # all-empty row
    assert np.isfinite(lat).all()


# ----------------------------------------------------- brute force agreement

def _random_tiny(seed, R=3, qlen=2, H=2, lens=(0, 1, 5)):
    g = torch.Generator().manual_seed(seed)
    total = sum(lens)
    pool = total + 4
    kv = (torch.randn(pool, 576, generator=g) * 0.5).to(torch.float8_e4m3fn).view(torch.uint8)
    perm = torch.randperm(pool, generator=g)[:total].to(torch.int32)
    indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q = torch.randn(R * qlen, H + 1, 576, generator=g).to(torch.bfloat16)
    w = (torch.randn(H, 128, 512, generator=g) / math.sqrt(512)).to(torch.bfloat16)
    gate = torch.randn(R * qlen, H * 128, generator=g).to(torch.bfloat16)
    return (bf16_bits(q), u8(kv), i32(perm), indptr, bf16_bits(w), bf16_bits(gate),
            np.array(lens, np.int32))


@pytest.mark.parametrize("seed", [0, 1])
def test_oracle_matches_brute_force(seed):
    q, kv, pages, indptr, w, gate, lens = _random_tiny(seed)
    scale, kvs, H, qlen = 1 / math.sqrt(192), 0.8, 2, 2
    lat, lse, out = O.decode_step(q, kv, pages, indptr, scale, kvs, H, qlen, w, gate, lens)
    blat, blse, bout = brute.decode_step(q, kv, pages, indptr, scale, kvs, H, qlen, w, gate)
    assert np.allclose(lat, np.array(blat), atol=1e-12, rtol=1e-12)
    b = np.array(blse)
    assert np.array_equal(np.isneginf(lse), np.isneginf(b))
    f = np.isfinite(b)
    assert np.allclose(lse[f], b[f], atol=1e-12)
    assert np.allclose(out, np.array(bout), atol=1e-12, rtol=1e-12)


# ------------------------------------------------------ absorbed = explicit

def test_absorbed_attention_equals_explicit_per_head_form():
    """Absorbed MLA (q_lat = W_UK^T q_nope over the 512-wide latent, W_UV
    after the attention) equals the explicit per-head form that up-projects
    each cached latent to a 128-dim key / value (``pre``: q_nope times W_UK
    gives the query's latent part; ``post``: W_UV applied to the latent)."""
    g = torch.Generator().manual_seed(4)
    H, L = 3, 17
    w_uk = (torch.randn(H, 128, 512, generator=g) / math.sqrt(512)).to(torch.bfloat16)
    w_uv = (torch.randn(H, 128, 512, generator=g) / math.sqrt(512)).to(torch.bfloat16)
    q_nope = torch.randn(H, 128, generator=g, dtype=torch.float64)
    q_pe = torch.randn(H, 64, generator=g, dtype=torch.float64)
    kv = (torch.randn(L, 576, generator=g) * 0.5).to(torch.float8_e4m3fn).view(torch.uint8)
    K = O.dequant(u8(kv), 0.8)
    c, k_pe = K[:, :512], K[:, 512:]
    Wk, Wv = O.bf16_to_f64(bf16_bits(w_uk)), O.bf16_to_f64(bf16_bits(w_uv))
    scale = 1 / math.sqrt(128 + 64)
    # explicit per head: keys [W_UK c ; k_pe], values W_UV c
    explicit = np.zeros((H, 128))
    for h in range(H):
        keys = np.concatenate([c @ Wk[h].T, k_pe], axis=1)           # [L, 192]
        vals = c @ Wv[h].T                                             # [L, 128]
        s = scale * keys @ np.concatenate([q_nope[h].numpy(), q_pe[h].numpy()])
        p = np.exp(s - s.max())
        explicit[h] = (p / p.sum()) @ vals
    # absorbed: one 576-dim query per head over the shared latent rows
    q576 = np.concatenate([np.einsum("hvc,hv->hc", Wk, q_nope.numpy()), q_pe.numpy()], 1)
    lat, _, _ = O.attend_rows(q576, K, scale)
    inf_gate = np.full((1, H * 128), 0x7F80, np.uint16)                # sigmoid(+inf) = 1
    out = O.value_gate(lat[None], bf16_bits(w_uv), inf_gate, np.array([L]), 1)
    assert np.allclose(out.reshape(H, 128), explicit, atol=1e-12, rtol=1e-10)


def test_value_gate_half_at_zero_gate():
    lat = O.bf16_to_f64(bf16_bits(W.make_latent(4, 2, seed=0)))
    w = W.make_inputs(0).w_uv[:2]
    zero = np.zeros((4, 256), np.uint16)
    inf = np.full((4, 256), 0x7F80, np.uint16)
    half = O.value_gate(lat, bf16_bits(w), zero, np.array([1, 1, 1, 1]), 1)
    full = O.value_gate(lat, bf16_bits(w), inf, np.array([1, 1, 1, 1]), 1)
    assert np.allclose(half * 2, full, atol=0, rtol=0)
    per_row = O.value_gate(lat, bf16_bits(w), inf, np.array([1, 0]), 2)
    assert np.all(per_row[2:] == 0) and np.array_equal(per_row[:2], full[:2])


# ------------------------------------------------------------- C oracle

def test_c_oracle_matches_numpy_oracle():
    from oracle import decode_step_c
    for inp in (W.make_inputs(0), W.make_inputs(4, lengths=[0, 3, 40, 1])):
        a = oracle_args(inp)
        extra = dict(w_uv_bits=bf16_bits(inp.w_uv), gate_bits=bf16_bits(inp.gate),
                     lengths=i32(inp.lengths))
        lat, lse, out = O.decode_step(**a, **extra)
        clat, clse, cout = decode_step_c(**a, w_uv_bits=extra["w_uv_bits"],
                                         gate_bits=extra["gate_bits"])
        assert np.allclose(clat, lat, atol=1e-12, rtol=1e-12)
        assert np.array_equal(np.isneginf(clse), np.isneginf(lse))
        f = np.isfinite(lse)
        assert np.allclose(clse[f], lse[f], atol=1e-12)
        assert np.allclose(cout, out, atol=1e-12, rtol=1e-12)


# --------------------------------------------------------- causal reading

def _spec_like(seed=3, R=3, qlen=4, H=2, lens=(2, 9, 40)):
    """Small speculative-decode inputs (qlen > 1), including a request shorter than qlen."""
    q, kv, pages, indptr, w, gate, lens = _random_tiny(seed, R=R, qlen=qlen, H=H, lens=lens)
    return dict(q_bits=q, kv_codes=kv, pages=pages, indptr=indptr, scale=1 / math.sqrt(192), kv_scale=0.8,
                heads=H, qlen=qlen), w, gate, lens


def test_causal_single_row_equals_unmasked():
    """With qlen 1 the causal reading shows every row all L_r tokens."""
    inp = W.make_inputs(0)
    a = oracle_args(inp)
    lat, lse = O.attend(**a)
    clat, clse = O.attend(**a, causal=True)
    assert np.array_equal(lat, clat) and np.array_equal(lse, clse)


def test_causal_row_equals_truncated_context():
    """Row tq of a request under the mask equals the unmasked attention of a
    request whose pages are cut to its first L - qlen + tq + 1 entries."""
    a, _, _, _ = _spec_like()
    qlen, H = a["qlen"], a["heads"]
    clat, clse = O.attend(**a, causal=True)
    R = len(a["indptr"]) - 1
    for r in range(R):
        lo, hi = int(a["indptr"][r]), int(a["indptr"][r + 1])
        L = hi - lo
        for tq in range(qlen):
            keep = max(0, L - qlen + tq + 1)
            t = r * qlen + tq
            pages = np.asarray(a["pages"][lo:lo + keep], np.int32)
            lat1, lse1 = O.attend(a["q_bits"][t:t + 1], a["kv_codes"], pages, np.array([0, keep], np.int32),
                                  a["scale"], a["kv_scale"], H, 1)
            assert np.allclose(clat[t], lat1[0], atol=1e-12, rtol=1e-12)
            if keep == 0:
                assert np.all(np.isneginf(clse[t])) and np.all(clat[t] == 0)
            else:
                assert np.allclose(clse[t], lse1[0], atol=1e-12)


def test_causal_matches_brute_force():
    a, w, gate, lens = _spec_like(seed=5)
    lat, lse, out = O.decode_step(**a, w_uv_bits=w, gate_bits=gate, lengths=lens, causal=True)
    blat, blse, bout = brute.decode_step(a["q_bits"], a["kv_codes"], a["pages"], a["indptr"], a["scale"],
                                         a["kv_scale"], a["heads"], a["qlen"], w, gate, causal=True)
    assert np.allclose(lat, np.array(blat), atol=1e-12, rtol=1e-12)
    b = np.array(blse)
    assert np.array_equal(np.isneginf(lse), np.isneginf(b))
    f = np.isfinite(b)
    assert np.allclose(lse[f], b[f], atol=1e-12)
    assert np.allclose(out, np.array(bout), atol=1e-12, rtol=1e-12)
    # the mask actually changes the early rows of the long request
    ulat, _ = O.attend(**a)
    assert not np.allclose(ulat[2 * 4], lat[2 * 4])


@pytest.mark.parametrize("ns,st", [(3, 4), (8, 5), (16, 1)])
def test_causal_merge_of_splits_equals_unsplit(ns, st):
    a, _, _, _ = _spec_like(seed=7)
    lat, lse = O.attend(**a, causal=True)
    o, ls = O.attend_splits(**a, num_splits=ns, split_tokens=st, causal=True)
    mlat, mlse = O.merge(o, ls)
    assert np.allclose(mlat, lat, atol=1e-12, rtol=1e-12)
    assert np.array_equal(np.isneginf(mlse), np.isneginf(lse))
    f = np.isfinite(lse)
    assert np.allclose(mlse[f], lse[f], atol=1e-12)


# ----------------------------------------------------- e4m3 encoder, KV append

def test_e4m3_encode_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = O.e4m3fn_to_f64(codes)
    assert np.array_equal(O.f64_to_e4m3fn(vals), codes)


def test_e4m3_encode_matches_torch_cast_in_range():
    g = torch.Generator().manual_seed(3)
    x = torch.cat([torch.randn(20000, generator=g) * s for s in (1e-3, 0.05, 1.0, 30.0, 150.0)])
    x = x[x.abs() <= 448]
    # every midpoint between adjacent representable values (ties to even)
    t = torch.from_numpy(O.e4m3fn_to_f64(np.arange(0x7F, dtype=np.uint8)))
    mids = ((t[1:] + t[:-1]) / 2).float()
    x = torch.cat([x, mids, -mids, torch.tensor([0.0, -0.0, 448.0, -448.0])])
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.f64_to_e4m3fn(x.double().numpy()), ref)


def test_e4m3_encode_saturates_and_keeps_nan():
    got = O.f64_to_e4m3fn(np.array([449.0, 464.0, 500.0, 1e30, np.inf, -np.inf, -1e6, np.nan, -np.nan]))
    assert got.tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F, 0x7F]
    # ties to even: 1.0625 lies halfway between 1.0 (0x38) and 1.125 (0x39)
    assert O.f64_to_e4m3fn(np.array([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -11])).tolist() == [0x38, 0x3A, 0x00, 0x01]


def test_kv_append_writes_the_slots_and_only_them():
    g = torch.Generator().manual_seed(9)
    pool, T = 40, 6
    kv = torch.randint(0, 255, (pool, 576), generator=g, dtype=torch.uint8).numpy()
    kv_c = (torch.randn(T, 512, generator=g) * 2).to(torch.bfloat16)
    k_pe = (torch.randn(T, 64, generator=g) * 2).to(torch.bfloat16)
    slots = np.array([3, -1, 17, 0, -5, 39], np.int64)
    ks = 0.8
    new = O.kv_append(kv, bf16_bits(kv_c), bf16_bits(k_pe), slots, ks)
    untouched = np.setdiff1d(np.arange(pool), slots[slots >= 0])
    assert np.array_equal(new[untouched], kv[untouched])
    for i, s in enumerate(slots):
        if s < 0:
            continue
        x = torch.cat([kv_c[i], k_pe[i]]).float() / ks            # float32 quotient
        assert np.array_equal(new[s], x.to(torch.float8_e4m3fn).view(torch.uint8).numpy())
    # read back through the decoder: within half an e4m3 step of the value
    back = O.dequant(new[slots[0]], ks)
    ref = torch.cat([kv_c[0], k_pe[0]]).double().numpy()
    assert np.all(np.abs(back - ref) <= np.abs(ref) * 2.0 ** -4 + 2.0 ** -10 * ks)


# ------------------------------------------------------------- block tables

@pytest.mark.parametrize("P", [2, 16, 64])
def test_block_table_rows_are_the_blocks_in_order(P):
    """Request rows under a block table: the concatenated row ranges of the
    request's blocks, cut to its length."""
    inp = W.make_block_inputs(4, "cpu", page_size=P, lengths=[0, 1, P, P + 1, 3 * P - 1, 200])
    pages, indptr = i32(inp.pages), i32(inp.indptr)
    last = i32(inp.extra["last_page_len"])
    lens = i32(inp.lengths)
    for r in range(len(lens)):
        blocks = pages[indptr[r]:indptr[r + 1]]
        want = [row for b in blocks for row in range(int(b) * P, int(b) * P + P)][:lens[r]]
        got = O.request_rows(pages, indptr, r, P, last)
        assert got.tolist() == want


@pytest.mark.parametrize("P", [4, 16])
def test_block_table_attention_equals_flat_page_list(P):
    inp = W.make_block_inputs(4, "cpu", page_size=P, lengths=[0, 5, 200, 333, 64])
    a = oracle_args(inp)
    last = i32(inp.extra["last_page_len"])
    lat, lse = O.attend(**a, page_size=P, last_page_len=last)
    rows = [O.request_rows(a["pages"], a["indptr"], r, P, last) for r in range(len(a["indptr"]) - 1)]
    flat_indptr = np.concatenate([[0], np.cumsum([len(x) for x in rows])]).astype(np.int32)
    flat = dict(a, pages=np.concatenate(rows).astype(np.int32), indptr=flat_indptr)
    lat1, lse1 = O.attend(**flat)
    assert np.array_equal(lat, lat1) and np.array_equal(lse, lse1)
    o, ls = O.attend_splits(**a, num_splits=5, split_tokens=50, page_size=P, last_page_len=last)
    o1, ls1 = O.attend_splits(**flat, num_splits=5, split_tokens=50)
    assert np.array_equal(ls, ls1) and np.array_equal(np.nan_to_num(o, nan=7.0), np.nan_to_num(o1, nan=7.0))


def _shard_by_slot(pages, indptr, ranks):
    """Decode-context-parallel sharding: token i of a request goes to rank
    i % ranks; returns each rank's (pages, indptr)."""
    out = []
    for k in range(ranks):
        pg, ip = [], [0]
        for r in range(len(indptr) - 1):
            own = pages[indptr[r]:indptr[r + 1]][k::ranks]
            pg.extend(own.tolist())
            ip.append(ip[-1] + len(own))
        out.append((np.array(pg, np.int32), np.array(ip, np.int32)))
    return out


@pytest.mark.parametrize("ranks", [2, 3])
def test_combine_of_sharded_partials_equals_full_attention(ranks):
    """The second-level LSE combine (``post``: the DCP combine of per-rank
    partials) is the same merge: attention over each rank's slice of the
    context, stacked as splits and merged, equals attention over it all."""
    inp = W.make_inputs(4, "cpu", lengths=[0, 5, 200, 333, 1])
    a = oracle_args(inp)
    lat, lse = O.attend(**a)
    parts_o, parts_l = [], []
    for pg, ip in _shard_by_slot(a["pages"], a["indptr"], ranks):
        o, l = O.attend_splits(**dict(a, pages=pg, indptr=ip), num_splits=2, split_tokens=64)
        parts_o.append(o)
        parts_l.append(l)
    mlat, mlse = O.merge(np.concatenate(parts_o), np.concatenate(parts_l))
    assert np.allclose(mlat, lat, atol=1e-12, rtol=1e-12)
    assert np.array_equal(np.isneginf(mlse), np.isneginf(lse))
    f = np.isfinite(lse)
    assert np.allclose(mlse[f], lse[f], atol=1e-12)


# ---------------------------------------------------------------- fp8 query

def test_fp8_query_equals_the_bf16_query_of_the_same_values():
    """An e4m3 query is exactly representable in bf16: attention over q8
    with scale s equals attention over bf16(q8 values) with scale s, and a
    q_scale folded into the scale equals scaling the query values."""
    inp = W.make_inputs(4, "cpu", lengths=[0, 5, 200, 33])
    a = oracle_args(inp)
    q8 = (inp.q.float() * 7).to(torch.float8_e4m3fn)          # some codes saturate, fine
    as_bf16 = q8.float().to(torch.bfloat16)
    assert torch.equal(as_bf16.float(), q8.float())               # exact widening
    lat8, lse8 = O.attend(**dict(a, q_bits=u8(q8.view(torch.uint8))), q_fp8=True)
    latb, lseb = O.attend(**dict(a, q_bits=bf16_bits(as_bf16)))
    assert np.array_equal(lat8, latb) and np.array_equal(lse8, lseb)
    qs = 0.25
    lat_s, lse_s = O.attend(**dict(a, q_bits=u8(q8.view(torch.uint8)), scale=a["scale"] * qs), q_fp8=True)
    scaled = (q8.float() * qs).to(torch.bfloat16)                 # exact: power-of-two scale
    lat_r, lse_r = O.attend(**dict(a, q_bits=bf16_bits(scaled)))
    assert np.allclose(lat_s, lat_r, atol=1e-12) and np.allclose(np.nan_to_num(lse_s, neginf=0),
                                                                 np.nan_to_num(lse_r, neginf=0), atol=1e-12)
