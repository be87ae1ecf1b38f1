"""Plain fp64 CPU oracle of the MLA paged decode step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module; the library
(``mla_decode_paged_gb300``) never does, and this module imports nothing from
it.  Inputs are numpy arrays of raw codes (uint8 fp8 codes, uint16 bf16
bits, int32 indices); every value is widened to float64 by the decoders
below, and every step is the plain definition, written out with no blocking,
fusion or reordering beyond it.

What the path computes, per request r, query row t (r*qlen <= t <
(r+1)*qlen) and real head h < H (vLLM API page
``vllm.models.kimi_k3.amd.specialized_decode.runtime.mla``, functions
``m1c_inputs`` and ``attend``; page
``vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.mla.value``, classes
``MlaValue`` and ``MlaGate``):

    K_j          = e4m3fn(kv[pages[indptr[r] + j]]) * kv_scale,  j < L_r
    s_j          = scale * <q[t, h, :576], K_j[:576]>
    lse[t, h]    = ln sum_j exp(s_j)                  (-inf when L_r == 0)
    latent[t, h] = sum_j exp(s_j - lse) * K_j[:512]   (0 when L_r == 0)
    val[t, h, v] = sum_c latent[t, h, c] * W_UV[h, v, c]
    out[t, h*128 + v] = val * sigmoid(gate[t, h*128 + v])  if L_r > 0 else 0

Readings where the pages are silent (each one is listed with its reason in
the design notes): no intra-request causal mask by default, and with
``causal=True`` row tq of a request sees only its first L_r - qlen + tq + 1
tokens (the speculative-decode convention: the request's last qlen tokens
are its own query positions); natural-log LSE of the
scaled scores; ``kv_scale`` multiplies the stored fp8 value and applies to
both the score K and the value V; OCP e4m3fn; page size 1; the split plan
of :func:`split_plan`; the gate is raw logits and the sigmoid is exact.
"""

from __future__ import annotations

import math

import numpy as np

D_QK = 576
D_LATENT = 512
D_V = 128


# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------

def e4m3fn_to_f64(codes) -> np.ndarray:
    """Decode OCP FP8 E4M3 ("e4m3fn") bytes to float64.

    The cache is read through ``current_platform.fp8_dtype()`` (``attend`` and
    ``m1c_inputs``: ``kv_cache.view(fp8)``); on this GPU that is OCP E4M3:
    1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, subnormals when
    the exponent field is 0, NaN for S.1111.111, no infinities.
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = sign * np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    subnormal = sign * np.ldexp(m / 8.0, -6)
    out = np.where(e == 0, subnormal, normal)
    out = np.where((e == 15) & ((c & 7) == 7), np.nan, out)
    return out.astype(np.float64)


def bf16_to_f64(bits) -> np.ndarray:
    """Widen bfloat16 bit patterns (uint16) to float64: a bf16 is the top half
    of an IEEE binary32, so the widening is exact."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def sigmoid(x) -> np.ndarray:
    """The logistic function 1 / (1 + exp(-x)), in float64.  ``MlaGate`` and
    ``MlaValue`` apply it to the raw gate inside the kernel."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-x))


# ---------------------------------------------------------------------------
# Paged gather
# ---------------------------------------------------------------------------

def request_rows(pages, indptr, r: int, page_size: int = 1, last_page_len=None) -> np.ndarray:
    """Row indices of request r's tokens in the KV pool, in order.

    Page size 1 (``m1c_inputs`` views the cache as one 576-wide row per
    token): ``pages[indptr[r]:indptr[r+1]]``.  Page size P > 1 (vLLM block tables): ``pages`` holds
    block indices and ``indptr`` counts blocks; block b covers rows
    [b*P, (b+1)*P); the request's last block holds ``last_page_len[r]``
    tokens, so L_r = (blocks - 1) * P + last_page_len[r] and token j is row
    ``pages[indptr[r] + j // P] * P + j % P``.
    """
    lo, hi = int(indptr[r]), int(indptr[r + 1])
    blocks = np.asarray(pages[lo:hi], dtype=np.int64)
    if page_size == 1:
        return blocks
    if blocks.size == 0:
        return blocks
    L = (blocks.size - 1) * page_size + int(last_page_len[r])
    j = np.arange(L, dtype=np.int64)
    return blocks[j // page_size] * page_size + j % page_size


def gather_rows(kv_codes, pages, indptr, r: int, page_size: int = 1, last_page_len=None) -> np.ndarray:
    """Request r's KV rows, as raw fp8 codes [L_r, 576]: the cache viewed as
    ``kv.view(-1, 576)``, one row per token, addressed through :func:`request_rows`
    (``m1c_inputs``: ``kv``, ``pages``, ``indptr``)."""
    kv_codes = np.asarray(kv_codes, dtype=np.uint8)
    return kv_codes[request_rows(pages, indptr, r, page_size, last_page_len)]


def gather_all(kv_codes, pages, indptr, page_size: int = 1, last_page_len=None) -> np.ndarray:
    """Every request's rows, concatenated in request order: [sum L, 576]."""
    R = len(indptr) - 1
    parts = [gather_rows(kv_codes, pages, indptr, r, page_size, last_page_len) for r in range(R)]
    if not parts:
        return np.zeros((0, D_QK), np.uint8)
    return np.concatenate(parts, axis=0)


# ---------------------------------------------------------------------------
# Attention of one request
# ---------------------------------------------------------------------------

def attend_rows(q_rows, K, scale: float, visible=None):
    """Softmax attention of query rows over one request's dequantised rows.

    ``q_rows``: float64 [n, 576] (n = qlen * H query rows of one request);
    ``K``: float64 [L, 576] (dequantised, kv_scale applied).  Multi-query
    form: every row attends over the same latent rows, keys are the full 576
    dims, values the first 512 (``attend``: forward_mqa on the latent cache).
    ``visible``: optional per-row count of leading rows of K the row may see
    (the causal mask); None means all L.

    Returns ``(latent [n, 512], lse [n], p [n, L])``; a row that sees no
    token gets latent 0, LSE -inf and p 0.
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    n = q_rows.shape[0]
    L = K.shape[0]
    vis = np.full(n, L, np.int64) if visible is None else np.clip(np.asarray(visible, np.int64), 0, L)
    latent = np.zeros((n, D_LATENT))
    lse = np.full(n, -np.inf)
    p = np.zeros((n, L))
    if L == 0:
        return latent, lse, p
    s = scale * (q_rows @ K.T)                       # [n, L]
    for i in range(n):
        v = int(vis[i])
        if v == 0:
            continue
        si = s[i, :v]
        m = si.max()
        e = np.exp(si - m)
        denom = e.sum()
        p[i, :v] = e / denom
        lse[i] = m + np.log(denom)
    # latent = p @ V, one matrix product per group of rows that see the same
    # number of tokens (every row at once without a mask)
    for v in np.unique(vis):
        if v == 0:
            continue
        sel = vis == v
        latent[sel] = p[sel, :v] @ K[:v, :D_LATENT]
    return latent, lse, p


def causal_visible(L: int, qlen: int, heads: int) -> np.ndarray:
    """Per query row (order (tq, h), as the rows of :func:`attend_rows`), the
    number of leading tokens it sees under the causal reading:
    L - qlen + tq + 1, clipped to [0, L]."""
    tq = np.repeat(np.arange(qlen, dtype=np.int64), heads)
    return np.clip(int(L) - qlen + tq + 1, 0, int(L))


_E4M3_TABLE = None


def dequant(codes, kv_scale: float) -> np.ndarray:
    """``e4m3fn(code) * kv_scale`` in float64 (the cache holds x / k_scale as
    fp8; ``m1c_inputs`` passes ``kv_scale=attn._k_scale_float``).  The codes
    are looked up in the 256 values :func:`e4m3fn_to_f64` gives (the same
    numbers, without its full-size temporaries)."""
    global _E4M3_TABLE
    if _E4M3_TABLE is None:
        _E4M3_TABLE = e4m3fn_to_f64(np.arange(256, dtype=np.uint8))
    return _E4M3_TABLE[np.asarray(codes, dtype=np.uint8)] * float(kv_scale)


def query_rows(q, t0: int, t1: int, heads: int, q_fp8: bool = False) -> np.ndarray:
    """Query rows t0..t1-1, real heads only, as float64 [(t1-t0)*heads, 576]:
    bf16 bits (the pages' q), or with ``q_fp8`` e4m3 codes (the DCP8 input
    ``q8``; its ``_q_scale`` multiplies the softmax scale, the caller folds
    it into ``scale``)."""
    blk = np.asarray(q)[t0:t1, :heads, :]
    vals = e4m3fn_to_f64(blk) if q_fp8 else bf16_to_f64(blk)
    return vals.reshape((t1 - t0) * heads, D_QK)


def attend(q_bits, kv_codes, pages, indptr, scale, kv_scale, heads, qlen,
           requests=None, return_p=False, causal=False, page_size=1, last_page_len=None, q_fp8=False):
    """The unsplit attention: latent [S, H, 512] and LSE [S, H].

    ``q_bits``: uint16 bf16 bits [S, H_pad, 576]; only heads < ``heads`` are
    read (``attend``: the real heads of a query padded 96 -> 128).
    ``requests``: optional subset of request indices to compute (others are
    left NaN), so that full-size workloads can be checked on a sample.
    ``causal``: apply :func:`causal_visible` to each request's rows.
    ``page_size`` / ``last_page_len``: block tables (:func:`request_rows`).
    ``q_fp8``: ``q_bits`` holds e4m3 codes (:func:`query_rows`).
    """
    q = np.asarray(q_bits)
    R = len(indptr) - 1
    S = R * qlen
    latent = np.full((S, heads, D_LATENT), np.nan)
    lse = np.full((S, heads), np.nan)
    ps = {}
    for r in (range(R) if requests is None else requests):
        K = dequant(gather_rows(kv_codes, pages, indptr, r, page_size, last_page_len), kv_scale)
        rows = query_rows(q, r * qlen, (r + 1) * qlen, heads, q_fp8)
        vis = causal_visible(K.shape[0], qlen, heads) if causal else None
        lat, l, p = attend_rows(rows, K, scale, vis)
        latent[r * qlen:(r + 1) * qlen] = lat.reshape(qlen, heads, D_LATENT)
        lse[r * qlen:(r + 1) * qlen] = l.reshape(qlen, heads)
        ps[r] = p.reshape(qlen, heads, -1)
    return (latent, lse, ps) if return_p else (latent, lse)


# ---------------------------------------------------------------------------
# Split-KV partials and their merge
# ---------------------------------------------------------------------------

def split_count(L: int, num_splits: int, split_tokens: int) -> int:
    """Splits request of length L is cut into: ceil(L / split_tokens), at
    least 1 and at most ``num_splits`` (the capacity of the partials' first
    dimension, ``m1c_inputs``: o [splits, S, 12, 512])."""
    if num_splits < 1 or split_tokens < 1:
        raise ValueError("num_splits and split_tokens must be >= 1")
    return max(1, min(num_splits, -(-int(L) // int(split_tokens))))


def split_plan(L: int, num_splits: int, split_tokens: int):
    """Token ranges [(start, end)] of a request's splits: n contiguous,
    near-equal ranges, the first ``L mod n`` one token longer.  The pages do
    not print the partition; this is the library's documented rule."""
    n = split_count(L, num_splits, split_tokens)
    base, rem = divmod(int(L), n)
    out = []
    start = 0
    for k in range(n):
        ln = base + (1 if k < rem else 0)
        out.append((start, start + ln))
        start += ln
    assert start == L
    return out


def attend_splits(q_bits, kv_codes, pages, indptr, scale, kv_scale, heads, qlen,
                  num_splits, split_tokens, requests=None, causal=False, page_size=1, last_page_len=None,
                  q_fp8=False, ranges=None):
    """Per-split partials: o [num_splits, S, H, 512] (float64) and lse
    [num_splits, S, H]; each used split is the attention restricted to its
    token range (``m1c_inputs``: new partials o [splits, S, 12, 512], LSE
    [splits, S, 12], merged afterwards).  Unused splits hold lse = -inf and
    o = NaN (their o is unspecified).  With ``causal``, a split's partial for
    a row covers the tokens of the split's range that the row sees; a row
    that sees none of them gets lse = -inf there.

    The pages fix the partials but not where a request is cut: by default
    the ranges are :func:`split_plan`'s; ``ranges`` (a mapping or sequence
    r -> [(start, end), ...], split k covering tokens start..end-1) gives
    them explicitly (``split_tokens`` is then unused)."""
    q = np.asarray(q_bits)
    R = len(indptr) - 1
    S = R * qlen
    o = np.full((num_splits, S, heads, D_LATENT), np.nan)
    lse = np.full((num_splits, S, heads), -np.inf)
    if requests is not None:
        lse[:] = np.nan
    for r in (range(R) if requests is None else requests):
        lse[:, r * qlen:(r + 1) * qlen] = -np.inf
        K = dequant(gather_rows(kv_codes, pages, indptr, r, page_size, last_page_len), kv_scale)
        rows = query_rows(q, r * qlen, (r + 1) * qlen, heads, q_fp8)
        vis = causal_visible(K.shape[0], qlen, heads) if causal else np.full(qlen * heads, K.shape[0])
        cuts = split_plan(K.shape[0], num_splits, split_tokens) if ranges is None else ranges[r]
        for k, (a, b) in enumerate(cuts):
            lat, l, _ = attend_rows(rows, K[a:b], scale, vis - a)
            if b > a:
                o[k, r * qlen:(r + 1) * qlen] = lat.reshape(qlen, heads, D_LATENT)
            lse[k, r * qlen:(r + 1) * qlen] = l.reshape(qlen, heads)
    return o, lse


def merge(o, lse):
    """LSE merge of split partials into the latent (``m1c_inputs``: "M1b
    merges the splits"; ``post``: the same LSE combine across DCP ranks).

        LSE    = ln sum_k exp(lse_k)
        latent = sum_k exp(lse_k - LSE) * o_k

    Splits with lse_k = -inf are skipped, never multiplied by 0 (their o is
    unspecified and may be NaN).  A row with every split empty gives latent
    0 and LSE -inf.
    """
    o = np.asarray(o, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    K = lse.shape[0]
    out_lse = np.full(lse.shape[1:], -np.inf)
    latent = np.zeros(o.shape[1:])
    valid = np.isfinite(lse)
    any_valid = valid.any(axis=0)
    m = np.where(valid, lse, -np.inf).max(axis=0)
    m_safe = np.where(any_valid, m, 0.0)
    total = np.zeros(lse.shape[1:])
    for k in range(K):
        w = np.where(valid[k], np.exp(np.where(valid[k], lse[k], 0.0) - m_safe), 0.0)
        total += w
        latent += np.where(valid[k][..., None], w[..., None] * np.nan_to_num(o[k], nan=0.0), 0.0)
    latent = np.where(any_valid[..., None], latent / np.where(any_valid, total, 1.0)[..., None], 0.0)
    out_lse = np.where(any_valid, m_safe + np.log(np.where(any_valid, total, 1.0)), -np.inf)
    return latent, out_lse


# ---------------------------------------------------------------------------
# Absorbed value up-projection and sigmoid gate
# ---------------------------------------------------------------------------

def value_gate(latent, w_uv_bits, gate_bits, lengths, qlen):
    """o_proj's input [S, H*128] (``post``: W_UV then the gate; ``MlaValue``
    / ``MlaGate``: value times the sigmoid of the raw gate, rows of empty
    requests zero).

    ``latent``: float64 [S, H, 512]; ``w_uv_bits``: bf16 bits [H, 128, 512]
    (latent axis contiguous, ``MlaValue``); ``gate_bits``: bf16 bits
    [S, H*128]; ``lengths``: per request; row t belongs to request t // qlen.
    Empty rows are selected to 0, never computed, so NaN gates do not leak.
    """
    latent = np.asarray(latent, dtype=np.float64)
    S, H, _ = latent.shape
    W = bf16_to_f64(w_uv_bits)                       # [H, 128, 512]
    val = np.einsum("thc,hvc->thv", latent, W)       # [S, H, 128]
    g = bf16_to_f64(gate_bits).reshape(S, H, D_V)
    lens = np.asarray(lengths).astype(np.int64)
    active = lens[np.arange(S) // qlen] > 0
    with np.errstate(invalid="ignore"):
        out = val * sigmoid(g)
    out = np.where(active[:, None, None], out, 0.0)
    return out.reshape(S, H * D_V)


def decode_step(q_bits, kv_codes, pages, indptr, scale, kv_scale, heads, qlen,
                w_uv_bits, gate_bits, lengths, requests=None, causal=False, page_size=1, last_page_len=None):
    """The whole step from raw inputs: (latent, lse, out).  With
    ``requests``, only those requests' rows are filled (the rest NaN)."""
    latent, lse = attend(q_bits, kv_codes, pages, indptr, scale, kv_scale, heads, qlen,
                         requests=requests, causal=causal, page_size=page_size, last_page_len=last_page_len)
    lat_in = np.nan_to_num(latent, nan=0.0)
    out = value_gate(lat_in, w_uv_bits, gate_bits, lengths, qlen)
    if requests is not None:
        keep = np.zeros(latent.shape[0], bool)
        for r in requests:
            keep[r * qlen:(r + 1) * qlen] = True
        out[~keep] = np.nan
    return latent, lse, out


# ---------------------------------------------------------------------------
# KV-cache append (the step that writes the cache the decode step reads)
# ---------------------------------------------------------------------------

_E4M3_POS = None


def _e4m3_positive_table():
    """The 127 non-negative finite E4M3 values (codes 0x00..0x7E), ascending."""
    global _E4M3_POS
    if _E4M3_POS is None:
        _E4M3_POS = e4m3fn_to_f64(np.arange(0x7F, dtype=np.uint8))
    return _E4M3_POS


def f64_to_e4m3fn(x) -> np.ndarray:
    """Encode float64 values as OCP E4M3 codes: round to the nearest
    representable value, ties to the even code (mantissa LSB 0); finite
    magnitudes above 448 and infinities saturate to +-448; NaN gives 0x7F.
    The sign of -0.0 and of negative values is kept.  (The cache write of
    the pages converts x / k_scale to fp8; the saturating conversion is this
    library's reading, the one CUDA's ``satfinite`` conversion makes.)"""
    x = np.asarray(x, dtype=np.float64)
    table = _e4m3_positive_table()
    a = np.abs(x)
    sat = np.where(np.isnan(a), 0.0, np.minimum(a, 448.0))
    hi = np.clip(np.searchsorted(table, sat, side="left"), 0, len(table) - 1)
    lo = np.clip(hi - 1, 0, len(table) - 1)
    d_hi = table[hi] - sat
    d_lo = sat - table[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(np.signbit(x), code | 0x80, code)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def kv_append(kv_codes, kv_c_bits, k_pe_bits, slots, k_scale: float) -> np.ndarray:
    """The cache after writing new tokens (vLLM API page
    ``vllm.models.kimi_k3.amd.specialized_decode.runtime.mla``, ``pre``:
    ``do_kv_cache_update`` stores the 512-wide ``kv_c`` and the 64-wide
    ``k_pe`` of each token, divided by ``k_scale`` and converted to fp8, at
    the token's slot, the row of the pool that attend later reads).

    ``kv_codes``: uint8 [pool, 576] (not modified; a copy is returned);
    ``kv_c_bits``: bf16 bits [T, 512]; ``k_pe_bits``: bf16 bits [T, 64];
    ``slots``: int64 [T], a negative slot skips its token (padding).  The
    quotient is taken in float32 (the precision the cache write computes
    in), then encoded by :func:`f64_to_e4m3fn`.
    """
    out = np.array(kv_codes, dtype=np.uint8, copy=True)
    rows = np.concatenate([bf16_to_f64(kv_c_bits), bf16_to_f64(k_pe_bits)], axis=1).astype(np.float32)
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        q = (rows / np.float32(k_scale)).astype(np.float64)
    codes = f64_to_e4m3fn(q)
    for i, s in enumerate(np.asarray(slots, np.int64)):
        if s >= 0:
            out[s] = codes[i]
    return out
