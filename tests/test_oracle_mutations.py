"""The oracle's pins catch plausible mistakes.  Each case plants one mistake
in the oracle (on the CPU, by patching one of its functions for the duration
of the test) and checks that at least one pin that does not compare against
another restatement of the method -- closed forms, the OCP table, torch's
casts, invariants of softmax attention and of the merge, the absorbed /
explicit identity -- then fails.  Nothing here touches the CUDA path."""

import math

import numpy as np
import pytest

from oracle import mla_oracle as O
from tests import test_oracle as T

# Pins tied to something other than the oracle itself, cheapest first.
PINS = [
    T.test_e4m3_ocp_table_values,
    T.test_e4m3_all_codes_match_torch_cast,
    T.test_bf16_decode_matches_torch,
    T.test_sigmoid_special_points,
    T.test_split_plan_golden,
    lambda: T.test_split_plan_partitions(1000, 7, 3),
    T.test_tiny_closed_form_golden,
    T.test_one_token_context_returns_that_row,
    T.test_softmax_weights_sum_to_one,
    T.test_constant_value_rows_give_that_row,
    T.test_zero_query_gives_mean_of_values,
    T.test_empty_request_zero_even_with_nan_gate,
    T.test_padded_heads_are_ignored,
    lambda: T.test_merge_of_splits_equals_unsplit(4, 25),
    T.test_merge_of_random_partition_equals_unsplit,
    lambda: T.test_merge_over_explicit_ranges_equals_unsplit(0),
    T.test_absorbed_attention_equals_explicit_per_head_form,
    T.test_value_gate_half_at_zero_gate,
    T.test_causal_single_row_equals_unmasked,
    T.test_causal_row_equals_truncated_context,
    T.test_e4m3_encode_round_trips_every_finite_code,
    T.test_e4m3_encode_matches_torch_cast_in_range,
    T.test_e4m3_encode_saturates_and_keeps_nan,
    T.test_kv_append_writes_the_slots_and_only_them,
    lambda: T.test_block_table_rows_are_the_blocks_in_order(16),
    lambda: T.test_block_table_attention_equals_flat_page_list(16),
    lambda: T.test_combine_of_sharded_partials_equals_full_attention(2),
    T.test_fp8_query_equals_the_bf16_query_of_the_same_values,
]


def _e4m3(bias=7, sub_exp=-6, nan=True):
    """An e4m3 decoder with one of its constants or rules changed."""
    def dec(codes):
        c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
        sign = np.where(c & 0x80, -1.0, 1.0)
        e, m = (c >> 3) & 0xF, (c & 0x7).astype(np.float64)
        out = np.where(e == 0, sign * np.ldexp(m / 8.0, sub_exp), sign * np.ldexp(1.0 + m / 8.0, e - bias))
        if nan:
            out = np.where((e == 15) & ((c & 7) == 7), np.nan, out)
        return out
    return dec


def _wrap_attend_rows(post):
    orig = O.attend_rows

    def f(q_rows, K, scale, visible=None):
        return post(orig, q_rows, K, scale, visible)
    return f


def _merge_without_skipping(o, lse):
    """LSE merge that weighs every split, multiplying an empty split's
    (unspecified, NaN) o by its zero weight."""
    o, lse = np.asarray(o, np.float64), np.asarray(lse, np.float64)
    m = np.max(lse, axis=0)
    m = np.where(np.isfinite(m), m, 0.0)
    w = np.exp(lse - m)
    tot = w.sum(0)
    return (w[..., None] * o).sum(0) / tot[..., None], m + np.log(tot)


def _value_gate_variant(row_of=lambda t, qlen: t // qlen, zero_empty=True, gate=None):
    def vg(latent, w_uv_bits, gate_bits, lengths, qlen):
        latent = np.asarray(latent, np.float64)
        S, H, _ = latent.shape
        val = np.einsum("thc,hvc->thv", latent, O.bf16_to_f64(w_uv_bits))
        g = O.bf16_to_f64(gate_bits).reshape(S, H, O.D_V)
        with np.errstate(invalid="ignore", over="ignore"):
            out = val * (O.sigmoid(g) if gate is None else gate(g))
        if zero_empty:
            active = np.asarray(lengths)[row_of(np.arange(S), qlen)] > 0
            out = np.where(active[:, None, None], out, 0.0)
        return out.reshape(S, H * O.D_V)
    return vg


def _split_plan_remainder_last(L, num_splits, split_tokens):
    n = O.split_count(L, num_splits, split_tokens)
    base, rem = divmod(int(L), n)
    lens = [base + (1 if k >= n - rem else 0) for k in range(n)]
    edges = np.concatenate([[0], np.cumsum(lens)]).astype(int).tolist()
    return list(zip(edges, edges[1:]))


def _request_rows_full_last_block(pages, indptr, r, page_size=1, last_page_len=None):
    lo, hi = int(indptr[r]), int(indptr[r + 1])
    blocks = np.asarray(pages[lo:hi], dtype=np.int64)
    if page_size == 1 or blocks.size == 0:
        return blocks
    j = np.arange(blocks.size * page_size, dtype=np.int64)
    return blocks[j // page_size] * page_size + j % page_size


def _query_rows_variant(from_pad=False, ignore_fp8=False):
    def qr(q, t0, t1, heads, q_fp8=False):
        q = np.asarray(q)
        blk = q[t0:t1, q.shape[1] - heads:, :] if from_pad else q[t0:t1, :heads, :]
        vals = O.e4m3fn_to_f64(blk) if (q_fp8 and not ignore_fp8) else O.bf16_to_f64(blk)
        return vals.reshape((t1 - t0) * heads, O.D_QK)
    return qr


def _merge_lse_without_max(merge):
    def f(o, lse):
        lat, out = merge(o, lse)
        m = np.max(np.where(np.isfinite(lse), lse, -np.inf), axis=0)
        return lat, np.where(np.isfinite(out), out - m, out)
    return f


def _mutations():
    """name -> (oracle function replaced, its replacement with the mistake)."""
    kv_append, encode, causal, dequant, merge = O.kv_append, O.f64_to_e4m3fn, O.causal_visible, O.dequant, O.merge
    vg = O.value_gate

    def enc_no_sat(x):
        c = encode(x)
        c[np.abs(np.asarray(x, np.float64)) > 464] = 0x7F
        return c

    return {
        "e4m3 exponent bias 8": ("e4m3fn_to_f64", _e4m3(bias=8)),
        "e4m3 subnormals scaled 2^-7": ("e4m3fn_to_f64", _e4m3(sub_exp=-7)),
        "e4m3 S.1111.111 decoded as a number": ("e4m3fn_to_f64", _e4m3(nan=False)),
        "bf16 widened from the wrong bit position": (
            "bf16_to_f64",
            lambda b: (np.asarray(b, np.uint16).astype(np.uint32) << 15).view(np.float32).astype(np.float64)),
        "sigmoid of -x": ("sigmoid", lambda x: 1.0 / (1.0 + np.exp(np.asarray(x, np.float64)))),
        "kv_scale dropped": ("dequant", lambda codes, kv_scale: dequant(codes, 1.0)),
        "kv_scale applied twice": ("dequant", lambda codes, kv_scale: dequant(codes, kv_scale) * kv_scale),
        "softmax scale dropped": ("attend_rows", _wrap_attend_rows(lambda f, q, K, s, v: f(q, K, 1.0, v))),
        "LSE in base 2": ("attend_rows", _wrap_attend_rows(
            lambda f, q, K, s, v: (lambda r: (r[0], r[1] / math.log(2), r[2]))(f(q, K, s, v)))),
        "rope dims dropped from the scores": ("attend_rows", _wrap_attend_rows(
            lambda f, q, K, s, v: f(np.concatenate([q[:, :512], 0 * q[:, 512:]], 1), K, s, v))),
        "values taken 64 dims late": ("attend_rows", _wrap_attend_rows(
            lambda f, q, K, s, v: (lambda r: (r[2] @ K[:, 64:576], r[1], r[2]))(f(q, K, s, v)))),
        "merge weighs empty splits": ("merge", _merge_without_skipping),
        "merge LSE without its max": ("merge", _merge_lse_without_max(merge)),
        "W_UV of the wrong head": ("value_gate", lambda lat, w, g, lens, ql: vg(lat, np.asarray(w)[::-1], g, lens,
                                                                               ql)),
        "gate used without the sigmoid": ("value_gate", _value_gate_variant(gate=lambda g: g)),
        "empty rows not zeroed": ("value_gate", _value_gate_variant(zero_empty=False)),
        "row t given to request t mod qlen": ("value_gate", _value_gate_variant(row_of=lambda t, ql: t % ql)),
        "split remainder given to the last splits": ("split_plan", _split_plan_remainder_last),
        "split count rounded down": ("split_count", lambda L, ns, st: max(1, min(ns, int(L) // int(st)))),
        "causal limit one token short": ("causal_visible", lambda L, ql, h: np.clip(causal(L, ql, h) - 1, 0, L)),
        "pad heads read instead of real heads": ("query_rows", _query_rows_variant(from_pad=True)),
        "fp8 query decoded as bf16": ("query_rows", _query_rows_variant(ignore_fp8=True)),
        "last block taken whole": ("request_rows", _request_rows_full_last_block),
        "KV append multiplies by k_scale": ("kv_append", lambda kv, c, p, s, ks: kv_append(kv, c, p, s, 1.0 / ks)),
        "e4m3 encode without saturation": ("f64_to_e4m3fn", enc_no_sat),
    }


MUTATIONS = _mutations()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_a_planted_mistake_fails_a_pin(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(O, attr, fn)
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except AssertionError:  # a pin's check failed (any other error would be a broken mutation)
            return
    pytest.fail("no pin caught: " + name)


def test_every_pin_passes_on_the_oracle_as_it_is():
    for pin in PINS:
        pin()
