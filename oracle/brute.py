"""Pure-Python brute force for tiny inputs: one routed (token, slot) at a time.

TEST INFRASTRUCTURE ONLY (imported by tests/ alone). It follows Eq. 13 of "Section 09: Grouped
GEMM" literally, row by row: the routed row is multiplied by its own expert's W_ug and W_down
(the "Grouped expert GEMM" page: each row uses its assigned expert's matrices), then weighted
and summed into its token ("grouped_mm" agent doc: scatter back and apply routing weights).
It never forms segments, offsets or a permutation, so it checks those independently.
"""
from __future__ import annotations

import math


def layer_forward(x, ids, weights, w_ug, w_down, E):
    """out[t] = sum over valid slots j of w[t][j] * SwiGLU(x[t] W_ug[e]^T) W_down[e]."""
    T, k = len(ids), len(ids[0])
    d = len(x[0])
    h = len(w_down[0])
    out = [[0.0] * d for _ in range(T)]
    for t in range(T):
        for j in range(k):
            e = int(ids[t][j])
            if e < 0 or e >= E:
                continue
            u = [sum(float(x[t][c]) * float(w_ug[e][r][c]) for c in range(d)) for r in range(2 * h)]
            a = [u[i] / (1.0 + math.exp(-u[i])) * u[h + i] for i in range(h)]
            y = [sum(a[i] * float(w_down[e][i][c]) for i in range(h)) for c in range(d)]
            wt = float(weights[t][j])
            for c in range(d):
                out[t][c] += wt * y[c]
    return out


def route(ids, E):
    """Counts, inclusive offsets and the stable placement by brute force: walk the experts in
    order and, for each, the flat slots in index order."""
    flat = [int(v) for row in ids for v in row]
    counts = [sum(1 for v in flat if v == e) for e in range(E)]
    offsets, run = [], 0
    for c in counts:
        run += c
        offsets.append(run)
    placed = []
    for e in range(E):
        for i, v in enumerate(flat):
            if v == e:
                placed.append(i)
    inv = [-1] * len(flat)
    for p, i in enumerate(placed):
        inv[i] = p
    return counts, offsets, placed, inv
