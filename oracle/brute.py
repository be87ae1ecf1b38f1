"""Pure-Python scalar brute force of the MLA decode step, for tiny inputs.

TEST INFRASTRUCTURE ONLY (same import rule as ``mla_oracle``).  It shares no
code with ``mla_oracle``: its own fp8 and bf16 decoders (``math.ldexp`` /
``struct`` on single codes), its own loops in place of matrix products, and
a two-pass softmax with ``math.exp`` / ``math.log``.  Tests run both on the
same tiny inputs and require agreement to ~1e-12, so an indexing, sign or
operand-order mistake in either one shows up.

Definitions followed: vLLM API pages
``vllm.models.kimi_k3.amd.specialized_decode.runtime.mla`` (``m1c_inputs``,
``attend``, ``post``) and
``vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.mla.value``
(``MlaValue``, ``MlaGate``).
"""

from __future__ import annotations

import math
import struct


def fp8_e4m3fn(code: int) -> float:
    """One OCP E4M3 byte to a Python float (bias 7, subnormals, S.1111.111 NaN)."""
    code &= 0xFF
    neg = code >= 128
    exp = (code >> 3) & 15
    man = code & 7
    if exp == 15 and man == 7:
        return math.nan
    if exp == 0:
        v = math.ldexp(man, -9)          # man/8 * 2^-6
    else:
        v = math.ldexp(8 + man, exp - 10)  # (1 + man/8) * 2^(exp-7)
    return -v if neg else v


def bf16(bits: int) -> float:
    """One bfloat16 bit pattern to a Python float."""
    return struct.unpack("<f", struct.pack("<I", (bits & 0xFFFF) << 16))[0]


def decode_step(q_bits, kv_codes, pages, indptr, scale, kv_scale, heads, qlen,
                w_uv_bits, gate_bits, dims=576, latent_dims=512, vdim=128, causal=False):
    """Nested loops over requests, rows, heads, tokens and dims.

    Inputs are nested Python sequences (or numpy arrays indexed one element
    at a time).  ``dims`` / ``latent_dims`` may be reduced for speed, the
    formula is the same.  With ``causal``, query row tq of a request with L
    tokens only sees token positions j <= L - qlen + tq.  Returns
    ``(latent, lse, out)`` as nested lists: latent[t][h][c], lse[t][h],
    out[t][h*vdim + v].
    """
    R = len(indptr) - 1
    latent, lse_out, out = [], [], []
    for r in range(R):
        start, stop = int(indptr[r]), int(indptr[r + 1])
        rows = []
        for i in range(start, stop):
            page = int(pages[i])
            rows.append([fp8_e4m3fn(int(kv_codes[page][d])) * kv_scale for d in range(dims)])
        for tq in range(qlen):
            t = r * qlen + tq
            lat_t, lse_t, out_t = [], [], []
            seen = rows
            if causal:
                last = len(rows) - qlen + tq          # last position this row may see
                seen = [row for j, row in enumerate(rows) if j <= last]
            for h in range(heads):
                qv = [bf16(int(q_bits[t][h][d])) for d in range(dims)]
                scores = []
                for row in seen:
                    acc = 0.0
                    for d in range(dims):
                        acc += qv[d] * row[d]
                    scores.append(scale * acc)
                if not seen:
                    lat = [0.0] * latent_dims
                    lse = -math.inf
                else:
                    mx = max(scores)
                    ssum = 0.0
                    for s in scores:
                        ssum += math.exp(s - mx)
                    lse = mx + math.log(ssum)
                    lat = [0.0] * latent_dims
                    for s, row in zip(scores, seen):
                        w = math.exp(s - lse)
                        for c in range(latent_dims):
                            lat[c] += w * row[c]
                lat_t.append(lat)
                lse_t.append(lse)
                for v in range(vdim):
                    if not rows:
                        out_t.append(0.0)
                        continue
                    acc = 0.0
                    for c in range(latent_dims):
                        acc += lat[c] * bf16(int(w_uv_bits[h][v][c]))
                    g = bf16(int(gate_bits[t][h * vdim + v]))
                    out_t.append(acc * (1.0 / (1.0 + math.exp(-g))))
            latent.append(lat_t)
            lse_out.append(lse_t)
            out.append(out_t)
    return latent, lse_out, out


def merge(o, lse):
    """Scalar LSE merge of split partials o[k][t][h][c], lse[k][t][h]: skip
    splits whose lse is -inf; all-empty rows give 0 and -inf."""
    K = len(lse)
    T = len(lse[0])
    H = len(lse[0][0])
    C = len(o[0][0][0])
    latent, out_lse = [], []
    for t in range(T):
        lt, ll = [], []
        for h in range(H):
            ks = [k for k in range(K) if lse[k][t][h] != -math.inf]
            if not ks:
                lt.append([0.0] * C)
                ll.append(-math.inf)
                continue
            mx = max(lse[k][t][h] for k in ks)
            tot = sum(math.exp(lse[k][t][h] - mx) for k in ks)
            big = mx + math.log(tot)
            row = [0.0] * C
            for k in ks:
                w = math.exp(lse[k][t][h] - big)
                for c in range(C):
                    row[c] += w * o[k][t][h][c]
            lt.append(row)
            ll.append(big)
        latent.append(lt)
        out_lse.append(ll)
    return latent, out_lse
