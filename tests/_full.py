"""Full-size oracle references for the GPU parity tests: each workload's
oracle result for every request is computed once per test session (the
inputs are drawn deterministically from the workload's seed on the device)
and shared by the tests that check different launches of that workload.
No arithmetic of the method here: the oracle computes, this module caches
and compares."""

import numpy as np

from oracle import mla_oracle as O
from tests._bits import bf16_bits, i32, u8
from tests.parity import assert_bf16_close, assert_lse_close, to_f64

_CACHE = {}


def reference(key, inp, *, causal=False, q_codes=None, q_scale=1.0, page_size=1, last_page_len=None,
              with_out=True):
    """(latent, lse, out) of the oracle for every request of ``inp`` (device
    tensors are copied to the host), cached under ``key``.  ``q_codes``: an
    fp8 query (uint8 codes) read with ``q_scale``; ``out`` is None when
    ``with_out`` is false."""
    if key in _CACHE:
        return _CACHE[key]
    blk = dict(page_size=page_size, last_page_len=None if last_page_len is None else i32(last_page_len))
    q_bits = bf16_bits(inp.q) if q_codes is None else u8(q_codes)
    a = dict(q_bits=q_bits, kv_codes=u8(inp.kv), pages=i32(inp.pages), indptr=i32(inp.indptr),
             scale=inp.scale * q_scale, kv_scale=inp.kv_scale, heads=inp.heads, qlen=inp.qlen)
    if with_out and q_codes is None:
        res = O.decode_step(**a, w_uv_bits=bf16_bits(inp.w_uv), gate_bits=bf16_bits(inp.gate),
                            lengths=i32(inp.lengths), causal=causal, **blk)
    else:
        lat, lse = O.attend(**a, causal=causal, q_fp8=q_codes is not None, **blk)
        res = (lat, lse, None)
    _CACHE[key] = res
    return res


def check_every_row(what, ref, latent, lse_m, out=None, capsys=None):
    """Element-wise parity of the merged LSE, latent and (optionally) out on
    every row; prints the largest LSE error and max|err|/max|ref| of each."""
    rlat, rlse, rout = ref
    e_lse = assert_lse_close(lse_m, rlse, what + ": lse")
    e_lat = assert_bf16_close(latent, rlat, what + ": latent")
    line = "%s: every row: max|lse err| %.3g, latent max|err|/max|ref| %.3g" % (
        what, e_lse, e_lat / max(float(np.abs(rlat).max()), 1e-300))
    if out is not None and rout is not None:
        e_out = assert_bf16_close(out, rout, what + ": out")
        line += ", out max|err|/max|ref| %.3g" % (e_out / max(float(np.abs(rout).max()), 1e-300))
    if capsys is not None:
        with capsys.disabled():
            print("\n[parity] " + line)
    return line


def as_f64(t):
    return to_f64(t)
