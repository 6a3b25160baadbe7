"""Pure-Python brute-force attention for tiny shapes (test infrastructure).

Nested lists and ``math.exp`` only -- no numpy, no library softmax -- so it
shares no code path with ``oracle.attention``.  It follows the per-head loop
of "step14_3 -- batched attention" (section "problem"): score every key,
drop the keys a mask excludes, exponentiate, normalise, and take the weighted
sum of the value rows.  Scores are not max-subtracted (the tiny test inputs
keep exp() in range), which is a different rounding path from the oracle.
"""

from __future__ import annotations

import math


def attend_one(q_row, keys, values, scale):
    """q_row [D]; keys, values: lists of [D] rows (already restricted)."""
    scores = []
    for k_row in keys:
        dot = 0.0
        for a, b in zip(q_row, k_row):
            dot += a * b
        scores.append(scale * dot)
    weights = [math.exp(s) for s in scores]
    total = sum(weights)
    D = len(values[0])
    out = [0.0] * D
    for w, v_row in zip(weights, values):
        for t in range(D):
            out[t] += (w / total) * v_row[t]
    return out


def decode(q, k_cache, v_cache, positions, scale):
    """q[b][h][D], caches[b][kvh][L][D] (nested lists, append already done)."""
    B, Hq, Hkv = len(q), len(q[0]), len(k_cache[0])
    g = Hq // Hkv
    out = []
    for b in range(B):
        P = int(positions[b])
        rows_b = []
        for h in range(Hq):
            kv = h // g
            keys = [k_cache[b][kv][j] for j in range(P + 1)]
            vals = [v_cache[b][kv][j] for j in range(P + 1)]
            rows_b.append(attend_one(q[b][h], keys, vals, scale))
        out.append(rows_b)
    return out


def decode_window(q, k_cache, v_cache, positions, scale, window):
    """As decode, over the last ``window`` rows up to each position only."""
    B, Hq, Hkv = len(q), len(q[0]), len(k_cache[0])
    g = Hq // Hkv
    out = []
    for b in range(B):
        P = int(positions[b])
        first = P - window + 1 if P - window + 1 > 0 else 0
        rows_b = []
        for h in range(Hq):
            kv = h // g
            keys = [k_cache[b][kv][j] for j in range(first, P + 1)]
            vals = [v_cache[b][kv][j] for j in range(first, P + 1)]
            rows_b.append(attend_one(q[b][h], keys, vals, scale))
        out.append(rows_b)
    return out


def prefill(q, k, v, start_pos, scale):
    """q[i][h][d] for new tokens; k, v [t][kvh][d] including the prefix."""
    S, Hq, Hkv = len(q), len(q[0]), len(k[0])
    g = Hq // Hkv
    out = []
    for i in range(S):
        row = []
        for h in range(Hq):
            kv = h // g
            last = start_pos + i
            keys = [k[j][kv] for j in range(last + 1)]
            vals = [v[j][kv] for j in range(last + 1)]
            row.append(attend_one(q[i][h], keys, vals, scale))
        out.append(row)
    return out
