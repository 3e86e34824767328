"""Tolerance comparison with mismatch counting.

TEST INFRASTRUCTURE (see the package docstring).  The checker's own behaviour
is pinned the way the Lesson K23 facts page (controls.checker) pins its
checker: a correct float32 result passes, the exact answer rounded to float32
passes, one output moved by more than the tolerance gives exactly one
mismatch, and zero tolerance rejects a float32 result.
"""

import numpy as np


def mismatches(got, want, atol):
    """Number of elements with |got - want| > atol.  NaN or inf in `got`
    where `want` is finite counts as a mismatch; -inf == -inf matches."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    if got.shape != want.shape:
        raise ValueError(f"shape mismatch {got.shape} vs {want.shape}")
    both_inf = np.isinf(got) & np.isinf(want) & (np.sign(got) == np.sign(want))
    diff = np.abs(got - want)
    bad = ~(diff <= atol) & ~both_inf
    return int(np.count_nonzero(bad))


def max_abs_err(got, want):
    """max |got - want| over finite pairs (inf where the two disagree on
    non-finite values, 0 for empty inputs)."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    if got.size == 0:
        return 0.0
    both_inf = np.isinf(got) & np.isinf(want) & (np.sign(got) == np.sign(want))
    diff = np.where(both_inf, 0.0, np.abs(got - want))
    if np.any(np.isnan(diff)):
        return float("inf")
    return float(diff.max())


def check(got, want, atol):
    """(ok, max_abs_err, mismatches)."""
    n = mismatches(got, want, atol)
    return n == 0, max_abs_err(got, want), n
