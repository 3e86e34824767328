"""Scalar-loop attention for tiny inputs: no matrix routines, no vectorisation.

TEST INFRASTRUCTURE (see the package docstring).  A second, independent
statement of the same definitions as oracle.attention ("Flash Attention 2 —
forward pass notes", section "The algorithm"; "Flash Attention 2 — backward
pass notes", section "The math (FA2 backward with recompute)"), written with
Python floats and math.exp so that a transposed operand or a dropped term in
the vectorised oracle shows up as a disagreement.  Use only for N, d <= ~8.
"""

import math


def _dot(a, b):
    s = 0.0
    for x, y in zip(a, b):
        s += float(x) * float(y)
    return s


def forward_head(q, k, v, scale, causal):
    """Returns (O as list of rows, LSE list) for one head; q, k, v [N][d]."""
    n = len(q)
    d = len(v[0])
    out, lse = [], []
    for i in range(n):
        scores = []
        for j in range(n):
            if causal and j > i:
                continue
            scores.append((j, scale * _dot(q[i], k[j])))
        m = max(s for _, s in scores)
        weights = [(j, math.exp(s - m)) for j, s in scores]
        l = sum(w for _, w in weights)
        row = [0.0] * d
        for j, w in weights:
            for c in range(d):
                row[c] += (w / l) * float(v[j][c])
        out.append(row)
        lse.append(m + math.log(l))
    return out, lse


def backward_head(q, k, v, do, scale, causal):
    """Returns (dQ, dK, dV) as lists of rows for one head."""
    n = len(q)
    d = len(q[0])
    # recompute P row by row
    p = [[0.0] * n for _ in range(n)]
    for i in range(n):
        vis = [j for j in range(n) if not (causal and j > i)]
        s = {j: scale * _dot(q[i], k[j]) for j in vis}
        m = max(s.values())
        l = sum(math.exp(x - m) for x in s.values())
        for j in vis:
            p[i][j] = math.exp(s[j] - m) / l
    o = [[sum(p[i][j] * float(v[j][c]) for j in range(n)) for c in range(d)]
         for i in range(n)]
    dq = [[0.0] * d for _ in range(n)]
    dk = [[0.0] * d for _ in range(n)]
    dv = [[0.0] * d for _ in range(n)]
    for i in range(n):
        d_i = _dot(do[i], o[i])
        for j in range(n):
            if p[i][j] == 0.0:
                continue
            dp = _dot(do[i], v[j])
            ds = p[i][j] * (dp - d_i)
            for c in range(d):
                dq[i][c] += ds * float(k[j][c]) * scale
                dk[j][c] += ds * float(q[i][c]) * scale
                dv[j][c] += p[i][j] * float(do[i][c])
    return dq, dk, dv
