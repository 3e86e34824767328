"""Softmax of one score row rounded to fp16, with and without the max subtracted.

TEST INFRASTRUCTURE (see the package docstring).  Restates the Lesson K23
facts page, block "overflow": in fp16 (largest finite 65504) exp(s) rounds to
infinity once s >= ln 65520; the naive softmax rounds exp, the sum and the
division each to fp16; the safe one subtracts the row max first.  Used to pin
why the kernels subtract the running max.
"""

import math

import numpy as np

FP16_OVERFLOW_THRESHOLD = math.log(65520.0)  # first value whose exp rounds to inf


def naive_fp16(row):
    """(weights, sum) with exp, sum and divide each rounded to fp16."""
    x = np.asarray(row, dtype=np.float64)
    e = np.exp(x).astype(np.float16)
    s = np.float16(0)
    for t in e:
        s = np.float16(s + t)
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        w = (e / s).astype(np.float16)
    return w, s


def safe_fp16(row):
    """(weights, sum) with the max subtracted before exp, then as naive_fp16."""
    x = np.asarray(row, dtype=np.float64)
    return naive_fp16(x - x.max())


def overflow_factor(row, lo=1.0, hi=16.0, iters=60):
    """Smallest factor f >= lo such that naive_fp16(f * row) has an infinite sum
    (bisection; assumes overflow at hi and monotone in f for positive maxima)."""
    x = np.asarray(row, dtype=np.float64)

    def overflows(f):
        with np.errstate(over="ignore"):
            return not np.isfinite(naive_fp16(f * x)[1])

    if overflows(lo):
        return lo
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if overflows(mid):
            hi = mid
        else:
            lo = mid
    return hi
