"""Pins of the split-KV oracle (oracle/split_kv.py): its merged result against
the plain definition (oracle/attention.py, an independent module), closed
forms for one-key slices, brute force, the merge's algebra (associative,
commutative, empty state neutral) and the rule for which slices a row reads.

Sources: "Flash Attention 2 — forward pass notes", section "Loop (per (b, h,
Q-tile))" (merging block states); Lesson K23 facts page,
`sources.onlineSoftmax.claims[2]` (associative, commutative merge)."""

import itertools

import numpy as np
import pytest

from oracle import attention as A
from oracle import brute
from oracle import split_kv as SK


def rand_head(n, d, seed, sigma=1.0):
    rng = np.random.default_rng(seed)
    return (rng.normal(0, sigma, (n, d)), rng.normal(0, sigma, (n, d)),
            rng.normal(0, 1, (n, d)))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,kps", [(1, 256), (7, 3), (200, 256), (256, 256), (600, 256),
                                   (600, 512), (513, 128), (50, 1)])
def test_merge_of_slices_is_attention(n, kps, causal):
    q, k, v = rand_head(n, 16, 100 + n + kps, sigma=2.0)
    scale = 0.25
    S = SK.num_slices(n, kps)
    o_parts = np.full((S, n, 16), np.nan)
    l_parts = np.full((S, n), np.nan)
    for s in range(S):
        o_s, l_s = SK.slice_head(q, k, v, scale, causal, s * kps, min(n, (s + 1) * kps))
        rows = [i for i in range(n) if SK.reads(i, s, kps, causal)]
        o_parts[s, rows], l_parts[s, rows] = o_s[rows], l_s[rows]
    o, lse = SK.merge_head(o_parts, l_parts, kps, causal)
    o_ref, lse_ref = A.forward_head(q, k, v, scale, causal)
    assert np.max(np.abs(o - o_ref)) < 1e-12
    assert np.max(np.abs(lse - lse_ref)) < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_read_rule_matches_visible_keys(causal):
    """L_s is finite exactly where the row reads the slice (sees one of its keys)."""
    n, kps = 300, 64
    q, k, v = rand_head(n, 8, 7)
    for s in range(SK.num_slices(n, kps)):
        _, l_s = SK.slice_head(q, k, v, 0.3, causal, s * kps, min(n, (s + 1) * kps))
        for i in range(n):
            assert np.isfinite(l_s[i]) == SK.reads(i, s, kps, causal)


def test_one_key_slices_closed_form():
    """With one key per slice, slice j of row i is (O = v_j, L = scale q_i.k_j)."""
    q, k, v = rand_head(5, 4, 3)
    scale = 0.7
    for j in range(5):
        o_s, l_s = SK.slice_head(q, k, v, scale, False, j, j + 1)
        assert np.array_equal(o_s, np.repeat(v[j][None, :], 5, axis=0))
        assert np.allclose(l_s, scale * (q @ k[j]), atol=0, rtol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_one_key_slices_against_brute_force(causal):
    """Merging one-key slices reproduces the scalar-loop attention."""
    n = 4
    q, k, v = rand_head(n, 3, 11)
    o_parts = np.zeros((n, n, 3))
    l_parts = np.zeros((n, n))
    for j in range(n):
        o_parts[j], l_parts[j] = SK.slice_head(q, k, v, 0.5, causal, j, j + 1)
    o, lse = SK.merge_head(o_parts, l_parts, 1, causal)
    o_b, lse_b = brute.forward_head(q, k, v, 0.5, causal)
    assert np.max(np.abs(o - np.asarray(o_b))) < 1e-14
    assert np.max(np.abs(lse - np.asarray(lse_b))) < 1e-14


def test_single_slice_is_identity():
    q, k, v = rand_head(90, 8, 5)
    o_s, l_s = SK.slice_head(q, k, v, 0.4, True, 0, 90)
    o, lse = SK.merge_head(o_s[None], l_s[None], 256, True)
    assert np.max(np.abs(o - o_s)) == 0.0
    assert np.max(np.abs(lse - l_s)) < 1e-15


def test_merge_order_and_bracketing():
    """Any order and any bracketing of the pairwise merge give the same state."""
    rng = np.random.default_rng(4)
    states = []
    for _ in range(4):
        m = rng.normal(0, 5, 6)
        states.append((m, rng.uniform(0.5, 3, 6), rng.normal(0, 1, (6, 2))))
    base = SK.finish(SK.merge_states(SK.merge_states(SK.merge_states(states[0], states[1]),
                                                     states[2]), states[3]))
    for perm in itertools.permutations(range(4)):
        st = [states[i] for i in perm]
        left = SK.merge_states(SK.merge_states(SK.merge_states(st[0], st[1]), st[2]), st[3])
        tree = SK.merge_states(SK.merge_states(st[0], st[1]), SK.merge_states(st[2], st[3]))
        for got in (SK.finish(left), SK.finish(tree)):
            assert np.max(np.abs(got[0] - base[0])) < 1e-13
            assert np.max(np.abs(got[1] - base[1])) < 1e-13


def test_empty_state_is_neutral_and_unread_entries_ignored():
    q, k, v = rand_head(40, 8, 9)
    o_s, l_s = SK.slice_head(q, k, v, 0.4, False, 0, 40)
    empty_o = np.full((40, 8), np.nan)      # never read: its L is -inf
    empty_l = np.full(40, -np.inf)
    o, lse = SK.merge_head(np.stack([empty_o, o_s, empty_o]), np.stack([empty_l, l_s, empty_l]),
                           40, False)
    assert np.max(np.abs(o - o_s)) < 1e-15 and np.max(np.abs(lse - l_s)) < 1e-15
    # causal: slices a row does not read may hold anything
    n, kps = 20, 8
    q, k, v = rand_head(n, 4, 10)
    S = SK.num_slices(n, kps)
    o_parts = np.full((S, n, 4), np.nan)
    l_parts = np.full((S, n), np.nan)
    for s in range(S):
        o_s, l_s = SK.slice_head(q, k, v, 0.4, True, s * kps, min(n, (s + 1) * kps))
        rows = [i for i in range(n) if SK.reads(i, s, kps, True)]
        o_parts[s, rows], l_parts[s, rows] = o_s[rows], l_s[rows]
    o, lse = SK.merge_head(o_parts, l_parts, kps, True)
    assert np.isfinite(o).all() and np.isfinite(lse).all()


def test_batched_partials_and_merge():
    rng = np.random.default_rng(12)
    q, k, v = (rng.normal(0, 1, (2, 70, 3, 8)) for _ in range(3))
    for causal in (False, True):
        op, lp = SK.partials(q, k, v, 0.35, causal, 32)
        o, lse = SK.merge(op, lp, 32, causal)
        o_ref, lse_ref = A.forward(q, k, v, 0.35, causal)
        assert np.max(np.abs(o - o_ref)) < 1e-12
        assert np.max(np.abs(lse - lse_ref)) < 1e-12
        # the entries of slices a row does not read are the NaN placeholders
        assert np.isnan(lp).any() == causal
