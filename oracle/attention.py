"""Plain float64 attention: the definition written out, one (batch, head) at a time.

TEST INFRASTRUCTURE (see the package docstring): only tests/, the smoke check
and the benchmark's CPU baseline may call this.

Sources
-------
* Forward: "Flash Attention 2 — forward pass notes", section "The algorithm":
  S = Q K^T / sqrt(d), causal mask S[i, j] = -inf for j > i, P = softmax(S)
  along each row, O = P V.  The scale is a caller argument (1/sqrt(d) in every
  workload here).
* Log-sum-exp saved for the backward: same page, section "What's still needed
  for full FA2", item 1: L = m_final + log(l_final), natural log of the scaled
  scores.
* Fully masked rows: same page, closing paragraph of that section, and
  "Flash Attention 2 — backward pass notes", section "Caveats specific to the
  backward path": a row whose every key is masked has l = 0, so L = -inf, the
  output row is zero and its gradient contributions are skipped.
* Backward: "Flash Attention 2 — backward pass notes", section "The math (FA2
  backward with recompute)": D = <dO, O> per row, P recomputed, dP = dO V^T,
  dS = P * (dP - D), dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO.

Layout of the batched entry points: q, k, v, dO, O and the gradients are
[B, N, H, d] (the pages' [B, T, C] with C = H * d, "Flash Attention 2 — forward
pass notes", section "Parity verification"); LSE and D are [B, H, N].

Everything is computed in float64 from whatever values are passed in (for the
bf16 workloads those are the bf16-rounded inputs read back exactly).
"""

import numpy as np


def _scores_head(q, k, scale, causal):
    """S = scale * Q K^T with the causal mask applied (j > i -> -inf)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    s = scale * (q @ k.T)
    if causal:
        n_q, n_k = s.shape
        i = np.arange(n_q)[:, None]
        j = np.arange(n_k)[None, :]
        s = np.where(j > i, -np.inf, s)
    return s


def probabilities_head(q, k, scale, causal):
    """Row-wise safe softmax of the masked scores, plus (m, l, LSE).

    Returns (P, m, l, lse), each float64.  m is the row max of the scaled
    scores, l = sum_j exp(S_ij - m_i), lse = m + log(l).  A row with no
    unmasked key has m = -inf, l = 0, P = 0 and lse = -inf.
    """
    s = _scores_head(q, k, scale, causal)
    m = s.max(axis=1)
    live = np.isfinite(m)
    e = np.zeros_like(s)
    e[live] = np.exp(s[live] - m[live, None])
    l = e.sum(axis=1)
    p = np.zeros_like(s)
    p[live] = e[live] / l[live, None]
    lse = np.full(m.shape, -np.inf)
    lse[live] = m[live] + np.log(l[live])
    return p, m, l, lse


def forward_head(q, k, v, scale, causal):
    """O = softmax(mask(scale Q K^T)) V and LSE for one (batch, head).

    q, k, v: [N, d].  Returns (O [N, d], LSE [N]) in float64.
    """
    p, _, _, lse = probabilities_head(q, k, scale, causal)
    o = p @ np.asarray(v, dtype=np.float64)
    return o, lse


def backward_head(q, k, v, do, scale, causal):
    """Analytic gradients of the float64 forward for one (batch, head).

    Returns dict with dq, dk, dv [N, d], and the intermediates the pins use:
    P, dP, dS, D (= rowsum(dO * O)), O and LSE.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    p, _, _, lse = probabilities_head(q, k, scale, causal)
    o = p @ v
    d_row = np.sum(do * o, axis=1)            # D_i = <dO_i, O_i>
    dv = p.T @ do                             # dV = P^T dO
    dp = do @ v.T                             # dP_ij = <dO_i, V_j>
    ds = p * (dp - d_row[:, None])            # dS = P * (dP - D)
    dq = scale * (ds @ k)                     # dQ = scale dS K
    dk = scale * (ds.T @ q)                   # dK = scale dS^T Q
    return {"dq": dq, "dk": dk, "dv": dv, "P": p, "dP": dp, "dS": ds,
            "D": d_row, "O": o, "lse": lse}


def _heads(x):
    """[B, N, H, d] -> iterator over (b, h, x[b, :, h, :])."""
    B, _, H, _ = x.shape
    for b in range(B):
        for h in range(H):
            yield b, h


def forward(q, k, v, scale, causal, heads=None):
    """Batched forward over [B, N, H, d] inputs.

    heads: optional iterable of (b, h) pairs to compute; the other rows of the
    outputs are left as NaN.  Returns (O [B, N, H, d], LSE [B, H, N]).
    """
    B, N, H, d = q.shape
    o = np.full((B, N, H, d), np.nan)
    lse = np.full((B, H, N), np.nan)
    for b, h in (heads if heads is not None else _heads(q)):
        o[b, :, h, :], lse[b, h, :] = forward_head(
            q[b, :, h, :], k[b, :, h, :], v[b, :, h, :], scale, causal)
    return o, lse


def backward(q, k, v, do, scale, causal, heads=None):
    """Batched backward over [B, N, H, d] inputs.

    Returns (dQ, dK, dV [B, N, H, d], D [B, H, N]); heads as in forward().
    """
    B, N, H, d = q.shape
    dq = np.full((B, N, H, d), np.nan)
    dk = np.full((B, N, H, d), np.nan)
    dv = np.full((B, N, H, d), np.nan)
    dd = np.full((B, H, N), np.nan)
    for b, h in (heads if heads is not None else _heads(q)):
        g = backward_head(q[b, :, h, :], k[b, :, h, :], v[b, :, h, :],
                          do[b, :, h, :], scale, causal)
        dq[b, :, h, :] = g["dq"]
        dk[b, :, h, :] = g["dk"]
        dv[b, :, h, :] = g["dv"]
        dd[b, h, :] = g["D"]
    return dq, dk, dv, dd
