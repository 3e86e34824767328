"""Split-KV attention: per-slice results over key slices, and their merge.

TEST INFRASTRUCTURE (see the package docstring).  Plain float64, one (batch,
head) at a time.  Independent of oracle.attention: it never calls it, and the
tests compare the merged result with that module's forward.

Sources
-------
* "Flash Attention 2 — forward pass notes", section "Loop (per (b, h,
  Q-tile))": the softmax of a concatenation of key blocks is the merge of the
  blocks' states.  A state is (m, l, O): m the max of the scaled scores seen,
  l = sum exp(s - m), O = sum exp(s - m) v (unnormalised).  Two states merge
  as m = max(m_a, m_b), l = l_a exp(m_a - m) + l_b exp(m_b - m),
  O = O_a exp(m_a - m) + O_b exp(m_b - m); the row's output is O / l and its
  log-sum-exp is m + log l.
* Lesson K23 facts page, `sources.onlineSoftmax.claims[2]`: the merge is
  associative and commutative, so the slices may be merged in any order and
  bracketing.

A slice result of row i over keys [lo, hi) is the attention of row i
restricted to those keys (with the causal mask j <= i by the keys' global
indices): O_s normalised over the slice and L_s = log sum exp of its scaled
scores; L_s = -inf when the row sees no key of the slice.  As a state it is
(m = L_s, l = 1, O = O_s), since exp(s - L_s) summed over the slice is 1.

Slices are [s * keys_per_split, (s + 1) * keys_per_split), s < ceil(N /
keys_per_split).  Row i reads slice s when it sees a key there: causal, iff
s * keys_per_split <= i; otherwise always.
"""

import numpy as np


def num_slices(n, keys_per_split):
    return -(-n // keys_per_split)


def reads(i, s, keys_per_split, causal):
    """Whether row i sees at least one key of slice s."""
    return (s * keys_per_split <= i) if causal else True


def slice_head(q, k, v, scale, causal, lo, hi):
    """Attention of every row of one head over the keys [lo, hi) alone.

    q: [Nq, d] for rows 0..Nq-1; k, v: [N, d].  Returns (O_s [Nq, d],
    L_s [Nq]); rows that see no key of the slice get O_s = 0, L_s = -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    ks = np.asarray(k, dtype=np.float64)[lo:hi]
    vs = np.asarray(v, dtype=np.float64)[lo:hi]
    s = scale * (q @ ks.T)
    if causal:
        i = np.arange(q.shape[0])[:, None]
        j = lo + np.arange(hi - lo)[None, :]
        s = np.where(j > i, -np.inf, s)
    o = np.zeros((q.shape[0], vs.shape[1]))
    lse = np.full(q.shape[0], -np.inf)
    if s.shape[1] == 0:
        return o, lse
    m = s.max(axis=1)
    live = np.isfinite(m)
    e = np.exp(s[live] - m[live, None])
    l = e.sum(axis=1)
    o[live] = (e @ vs) / l[:, None]
    lse[live] = m[live] + np.log(l)
    return o, lse


def merge_states(a, b):
    """The pairwise merge of two (m, l, O) states (O unnormalised, [rows, d]).

    m and l are [rows]; the empty state of a row is (-inf, 0, 0).
    """
    m_a, l_a, o_a = a
    m_b, l_b, o_b = b
    m = np.maximum(m_a, m_b)
    live = np.isfinite(m)
    wa = np.zeros_like(m)
    wb = np.zeros_like(m)
    wa[live] = np.exp(m_a[live] - m[live])
    wb[live] = np.exp(m_b[live] - m[live])
    return m, l_a * wa + l_b * wb, o_a * wa[:, None] + o_b * wb[:, None]


def state_of(o_s, lse_s):
    """A slice result (O_s normalised, L_s) as a state (m = L_s, l = 1, O = O_s);
    rows with L_s = -inf become the empty state."""
    live = np.isfinite(lse_s)
    l = np.where(live, 1.0, 0.0)
    o = np.where(live[:, None], o_s, 0.0)
    return np.asarray(lse_s, dtype=np.float64), l, o


def finish(state):
    """(O, L) of a merged state: O / l, m + log l; O = 0, L = -inf where l = 0."""
    m, l, o = state
    live = l > 0
    out = np.zeros_like(o)
    out[live] = o[live] / l[live, None]
    lse = np.full(m.shape, -np.inf)
    lse[live] = m[live] + np.log(l[live])
    return out, lse


def merge_head(o_parts, lse_parts, keys_per_split, causal, order=None):
    """Merge one head's slice results, folding the states left to right.

    o_parts: [S, N, d]; lse_parts: [S, N].  Row i takes only the slices it
    reads (entries of the others are never looked at, whatever they hold).
    order: optional permutation of the slices.  Returns (O [N, d], L [N]).
    """
    S, N, d = o_parts.shape
    rows = np.arange(N)
    acc = (np.full(N, -np.inf), np.zeros(N), np.zeros((N, d)))
    for s in (order if order is not None else range(S)):
        use = np.array([reads(i, s, keys_per_split, causal) for i in rows])
        lse_s = np.where(use, lse_parts[s], -np.inf)
        o_s = np.where(use[:, None], o_parts[s], 0.0)
        acc = merge_states(acc, state_of(o_s, lse_s))
    return finish(acc)


def partials(q, k, v, scale, causal, keys_per_split, heads=None):
    """Batched slice results over [B, N, H, d] inputs.

    Returns (o_part [S, B, N, H, d], lse_part [S, B, H, N]); entries of rows
    that do not read a slice are NaN (they are never written or read).
    """
    B, N, H, d = q.shape
    S = num_slices(N, keys_per_split)
    o_part = np.full((S, B, N, H, d), np.nan)
    lse_part = np.full((S, B, H, N), np.nan)
    hs = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in hs:
        for s in range(S):
            lo, hi = s * keys_per_split, min(N, (s + 1) * keys_per_split)
            o_s, l_s = slice_head(q[b, :, h, :], k[b, :, h, :], v[b, :, h, :], scale, causal,
                                  lo, hi)
            rows = np.array([reads(i, s, keys_per_split, causal) for i in range(N)])
            o_part[s, b, rows, h, :] = o_s[rows]
            lse_part[s, b, h, rows] = l_s[rows]
    return o_part, lse_part


def merge(o_part, lse_part, keys_per_split, causal, heads=None):
    """Batched merge: (O [B, N, H, d], L [B, H, N]) from the slice results."""
    S, B, N, H, d = o_part.shape
    o = np.full((B, N, H, d), np.nan)
    lse = np.full((B, H, N), np.nan)
    hs = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in hs:
        o[b, :, h, :], lse[b, h, :] = merge_head(o_part[:, b, :, h, :], lse_part[:, b, h, :],
                                                 keys_per_split, causal)
    return o, lse
