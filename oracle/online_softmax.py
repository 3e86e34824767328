"""Online-softmax restatement (running max m, running sum l, rescale alpha).

TEST INFRASTRUCTURE (see the package docstring).  This module is independent of
oracle.attention: it never calls it, and the tests compare the two.

Sources
-------
* "Flash Attention 2 — forward pass notes", sections "Notation" and "Loop (per
  (b, h, Q-tile))": per Q row keep m (running max of the scaled scores), l
  (running denominator) and O (unnormalised output); for each K block take the
  block max, m_new = max(m, m_block), alpha = exp(m - m_new), rescale O and l
  by alpha, then add exp(s - m_new) to l and exp(s - m_new) * V_j to O; finally
  O /= l.  Out-of-range and above-diagonal positions score -inf; with the
  causal mask, blocks that start after the tile's last row are skipped.
* Lesson K23 facts page, sources.onlineSoftmax (Milakov and Gimelshein,
  Algorithm 3): element-by-element m_j = max(m_{j-1}, x_j),
  d_j = d_{j-1} exp(m_{j-1} - m_j) + exp(x_j - m_j), m_0 = -inf, d_0 = 0; and
  the (m, d) pairs merge with an associative, commutative operator.
* Same page, controls.vector / correctness: the "broken" variant drops the
  rescale by alpha and is wrong whenever the running max rises after the first
  tile.
"""

import numpy as np


def merge(a, b):
    """Merge two (m, l) states: the pair for the concatenation of their inputs.

    (m_a, l_a) + (m_b, l_b) = (m, l_a exp(m_a - m) + l_b exp(m_b - m)),
    m = max(m_a, m_b).  The empty state is (-inf, 0).
    """
    m_a, l_a = a
    m_b, l_b = b
    m = max(m_a, m_b)
    if m == -np.inf:
        return (-np.inf, 0.0)
    return (m, l_a * np.exp(m_a - m) + l_b * np.exp(m_b - m))


def trace(values, tile=1, broken=False):
    """(m, l) after each tile of `tile` consecutive values of one score row.

    With tile=1 this is Algorithm 3 element by element.  broken=True omits the
    rescale of the old sum when the max rises (the old l is kept as it was).
    Returns a list of (m, l) floats, one per tile.
    """
    x = np.asarray(values, dtype=np.float64)
    m, l = -np.inf, 0.0
    out = []
    for t0 in range(0, x.size, tile):
        blk = x[t0:t0 + tile]
        m_new = max(m, float(blk.max()))
        alpha = 1.0 if broken else (np.exp(m - m_new) if m != -np.inf else 0.0)
        l = l * alpha + float(np.sum(np.exp(blk - m_new)))
        m = m_new
        out.append((m, l))
    return out


def max_rises(values):
    """How many times the running max rises after the first element."""
    x = np.asarray(values, dtype=np.float64)
    run = np.maximum.accumulate(x)
    return int(np.count_nonzero(run[1:] > run[:-1]))


def two_pass_weights(values):
    """Safe softmax of one row: max, then sum, then divide."""
    x = np.asarray(values, dtype=np.float64)
    e = np.exp(x - x.max())
    return e / e.sum()


def online_weights(values, tile=1):
    """Softmax weights from the final (m, l) of the online recurrence."""
    x = np.asarray(values, dtype=np.float64)
    m, l = trace(x, tile)[-1]
    return np.exp(x - m) / l


def tiled_attention_head(q, k, v, scale, causal, br, bc, broken=False,
                         dtype=np.float64):
    """FA2 loop order for one head: outer loop over Q tiles, inner over K blocks.

    q, k, v: [N, d].  br, bc: Q-tile and K-block sizes.  Arithmetic runs in
    `dtype` (float64 for the oracle's self-checks; float32 to restate a float32
    kernel's error).  Returns (O [N, d], LSE [N], traces) where traces[i] is
    the list of (m, l) after each K block visited by row i.
    """
    q = np.asarray(q, dtype=dtype)
    k = np.asarray(k, dtype=dtype)
    v = np.asarray(v, dtype=dtype)
    sc = dtype(scale)
    n, d = q.shape
    o_out = np.zeros((n, d), dtype=dtype)
    lse = np.zeros(n, dtype=np.float64)
    traces = [[] for _ in range(n)]
    for q0 in range(0, n, br):
        rows = range(q0, min(q0 + br, n))
        q_end = min(q0 + br, n) - 1           # last row of this Q tile
        m = {i: dtype(-np.inf) for i in rows}
        l = {i: dtype(0) for i in rows}
        acc = {i: np.zeros(d, dtype=dtype) for i in rows}
        for k0 in range(0, n, bc):
            if causal and k0 > q_end:          # causal block skip
                break
            cols = np.arange(k0, min(k0 + bc, n))
            for i in rows:
                s = (q[i] @ k[cols].T) * sc
                if causal:
                    s = np.where(cols > i, dtype(-np.inf), s)
                m_blk = s.max()
                m_new = max(m[i], m_blk)
                if m_new == -np.inf:            # nothing visible yet
                    traces[i].append((float(m[i]), float(l[i])))
                    continue
                if not broken:
                    alpha = dtype(np.exp(m[i] - m_new)) if m[i] != -np.inf else dtype(0)
                    acc[i] = acc[i] * alpha
                    l[i] = l[i] * alpha
                p = np.exp(s - m_new).astype(dtype)
                l[i] = l[i] + p.sum(dtype=dtype)
                acc[i] = acc[i] + (p @ v[cols]).astype(dtype)
                m[i] = m_new
                traces[i].append((float(m[i]), float(l[i])))
        for i in rows:
            if l[i] > 0:
                o_out[i] = acc[i] / l[i]
                lse[i] = float(m[i]) + np.log(float(l[i]))
            else:                              # fully masked row
                o_out[i] = 0
                lse[i] = -np.inf
    return o_out, lse, traces
