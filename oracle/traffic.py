"""Closed-form global-traffic and work counts of one attention head.

TEST INFRASTRUCTURE (see the package docstring).  Restates the Lesson K23 facts
page, block "traffic": with G = ceil(N / B) query blocks of B rows, the
unfused kernels (scores, row softmax, P V; Algorithm 0 of the FlashAttention
paper as quoted in sources.flashAttention) read N d + 2 G N d + 2 N^2 and
write 2 N^2 + N d four-byte elements; the fused kernel reads N d + 2 G N d and
writes N d.  The fused kernel takes one exp per score plus one rescale exp per
row per key block (N^2 + N G), and 2 N^2 d multiply-adds in either form.

These are the counts the benchmark's algorithmic-byte figures are checked
against (the fused kernel's unavoidable traffic is its N d + ... terms with
G = 1).
"""

import math


def counts(N, d, B, kind):
    """Dict of globalReads, globalWrites (elements), globalBytes (4-byte
    elements), extraMemoryBytes, fma and exps for one head."""
    G = math.ceil(N / B)
    if kind == "unfused":
        reads = N * d + 2 * G * N * d + 2 * N * N
        writes = 2 * N * N + N * d
        extra = 4 * N * N
        exps = N * N
    elif kind == "fused":
        reads = N * d + 2 * G * N * d
        writes = N * d
        extra = 0
        exps = N * N + N * G
    else:
        raise ValueError(kind)
    return {"globalReads": reads, "globalWrites": writes,
            "globalBytes": 4 * (reads + writes), "extraMemoryBytes": extra,
            "fma": 2 * N * N * d, "exps": exps}
