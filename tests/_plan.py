"""Decoding of attend work plans (layout in mla_decode.h, mla_plan_units)
for the tests: per-CTA items and per-request split ranges."""

import numpy as np

ITEM_WORDS = 4


def items(plan):
    """(G, offsets, items [n, 6] = r, k, n_r, group, start, count).  The
    plan ends with a copy of each CTA's first item (G x ITEM_WORDS words,
    zeros for a CTA without items); it is checked against the items."""
    p = np.asarray(plan, dtype=np.int64)
    G = int(p[0])
    off = p[1:G + 2]
    raw = p[G + 2:p.size - ITEM_WORDS * G].reshape(-1, ITEM_WORDS)
    first = p[p.size - ITEM_WORDS * G:].reshape(G, ITEM_WORDS)
    for b in range(G):
        want = raw[off[b]] if off[b] < off[b + 1] else np.zeros(ITEM_WORDS, dtype=np.int64)
        assert np.array_equal(first[b], want), "first-item copy of CTA %d" % b
    w = raw[:, 1]
    dec = np.stack([raw[:, 0], w & 511, (w >> 9) & 511, (w >> 18) & 8191, raw[:, 2], raw[:, 3]], axis=1)
    return G, off, dec


def ranges(plan, num_requests, group=0):
    """Per request, the token ranges [(start, end)] of its splits k = 0..n_r-1
    for one row group."""
    _, _, it = items(plan)
    out = [dict() for _ in range(num_requests)]
    for r, k, nr, g, s, c in it.tolist():
        if g == group:
            assert k not in out[r], "split %d of request %d twice" % (k, r)
            out[r][k] = (s, s + c, nr)
    res = []
    for r, d in enumerate(out):
        nr = {v[2] for v in d.values()}
        assert len(nr) == 1 and sorted(d) == list(range(nr.pop())), "request %d splits incomplete" % r
        res.append([(d[k][0], d[k][1]) for k in sorted(d)])
    return res
