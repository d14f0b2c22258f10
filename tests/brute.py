"""Pure-Python brute-force attention on contiguous K/V (no paging at all).

Used only to pin the oracle on tiny inputs: it never sees a block table, a
pool or a slot, so a gather mistake in the oracle cannot hide behind it.
Plain lists and ``math.exp``; causal rule: query j of a request whose first
new token sits at absolute position ctx sees keys 0 .. ctx + j.
"""
from __future__ import annotations

import math


def attend_one(qrow, keys, values, scale):
    """softmax(scale * q.k) weighted sum of values for one query row."""
    scores = [scale * sum(a * b for a, b in zip(qrow, k)) for k in keys]
    top = max(scores)
    weights = [math.exp(s - top) for s in scores]
    total = sum(weights)
    dim = len(values[0])
    return [sum(w * v[d] for w, v in zip(weights, values)) / total for d in range(dim)]


def attention(q_rows, k_seq, v_seq, ctx, num_kv_heads, scale):
    """One request.

    q_rows[j][h] -> list of floats (query j, query head h);
    k_seq[p][kv], v_seq[p][kv] -> list of floats (logical position p);
    returns out[j][h] lists.
    """
    n_heads = len(q_rows[0]) if q_rows else 0
    group = n_heads // num_kv_heads
    out = []
    for j, row in enumerate(q_rows):
        last = ctx + j
        out_row = []
        for h in range(n_heads):
            kv = h // group
            keys = [k_seq[p][kv] for p in range(last + 1)]
            vals = [v_seq[p][kv] for p in range(last + 1)]
            out_row.append(attend_one(row[h], keys, vals, scale))
        out.append(out_row)
    return out
