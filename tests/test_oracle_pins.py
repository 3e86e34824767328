"""Pins of the float64 oracle against facts that do not come from the oracle.

Each test names what it checks and where the fact comes from: a value printed
on the pages (tests/golden/), a closed form, an invariant of the mathematics,
a library routine for a special case, brute force, or finite differences.
"""

import math

import numpy as np
import pytest
from scipy import special

from oracle import attention as A
from oracle import brute, checker, fp16_softmax, online_softmax as OS, traffic


def _rand(rng, *shape, sigma=1.0):
    return rng.normal(0.0, sigma, size=shape)


# ---------------------------------------------------------------------------
# Definition-level pins (closed forms, invariants, library special cases)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_rows_of_p_sum_to_one(causal):
    rng = np.random.default_rng(1)
    q, k = _rand(rng, 37, 8), _rand(rng, 37, 8)
    p, _, _, _ = A.probabilities_head(q, k, 0.35, causal)
    assert np.max(np.abs(p.sum(axis=1) - 1.0)) < 1e-15
    if causal:
        assert np.all(p[np.triu_indices(37, 1)] == 0.0)


@pytest.mark.parametrize("causal", [False, True])
def test_softmax_and_lse_match_scipy(causal):
    """P and LSE against scipy.special.softmax / logsumexp of the masked scores."""
    rng = np.random.default_rng(2)
    n, d, scale = 29, 16, 0.25
    q, k = _rand(rng, n, d), _rand(rng, n, d)
    s = scale * (q @ k.T)
    if causal:
        s[np.triu_indices(n, 1)] = -np.inf
    p, m, l, lse = A.probabilities_head(q, k, scale, causal)
    np.testing.assert_allclose(p, special.softmax(s, axis=1), rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, special.logsumexp(s, axis=1), rtol=1e-15, atol=1e-13)


def test_causal_first_row_is_v0_and_its_dq_is_zero():
    rng = np.random.default_rng(3)
    n, d = 12, 8
    q, k, v, do = (_rand(rng, n, d) for _ in range(4))
    o, lse = A.forward_head(q, k, v, 0.3, True)
    assert np.array_equal(o[0], v[0])                 # P[0, 0] = 1 exactly
    assert lse[0] == 0.3 * float(q[0] @ k[0])         # log(1) = 0
    g = A.backward_head(q, k, v, do, 0.3, True)
    assert np.max(np.abs(g["dq"][0])) < 1e-15         # dS_00 = dP_00 - D_0 = 0


@pytest.mark.parametrize("causal", [False, True])
def test_single_key(causal):
    rng = np.random.default_rng(4)
    q, k, v, do = (_rand(rng, 1, 5) for _ in range(4))
    o, lse = A.forward_head(q, k, v, 0.7, causal)
    assert np.array_equal(o, v)
    assert lse[0] == pytest.approx(0.7 * float(q[0] @ k[0]), abs=1e-15)
    g = A.backward_head(q, k, v, do, 0.7, causal)
    np.testing.assert_allclose(g["dv"], do, atol=1e-15)
    assert np.max(np.abs(g["dq"])) < 1e-15 and np.max(np.abs(g["dk"])) < 1e-15


@pytest.mark.parametrize("causal", [False, True])
def test_scale_zero_gives_running_mean(causal):
    """scale = 0: every visible key weighs the same, so O_i is the mean of the
    visible V rows and LSE_i = log(#visible keys)."""
    rng = np.random.default_rng(5)
    n, d = 17, 6
    q, k, v = (_rand(rng, n, d) for _ in range(3))
    o, lse = A.forward_head(q, k, v, 0.0, causal)
    if causal:
        want = np.cumsum(v, axis=0) / np.arange(1, n + 1)[:, None]
        want_lse = np.log(np.arange(1, n + 1))
    else:
        want = np.broadcast_to(v.mean(axis=0), (n, d))
        want_lse = np.full(n, np.log(n))
    np.testing.assert_allclose(o, want, atol=1e-14)
    np.testing.assert_allclose(lse, want_lse, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_invariants(causal):
    """Rows of dS sum to zero (so sum_j dK_j = 0); sum_j dV_j = sum_i dO_i;
    D_i = <dO_i, O_i> equals sum_j P_ij dP_ij."""
    rng = np.random.default_rng(6)
    n, d = 23, 7
    q, k, v, do = (_rand(rng, n, d) for _ in range(4))
    g = A.backward_head(q, k, v, do, 0.4, causal)
    assert np.max(np.abs(g["dS"].sum(axis=1))) < 1e-13
    assert np.max(np.abs(g["dk"].sum(axis=0))) < 1e-12
    np.testing.assert_allclose(g["dv"].sum(axis=0), do.sum(axis=0), atol=1e-12)
    np.testing.assert_allclose(g["D"], np.sum(g["P"] * g["dP"], axis=1), atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_shift_invariance(causal):
    """K -> K + u (same u for every key) adds scale * q_i . u to every score of
    row i: O is unchanged and LSE_i moves by exactly that amount."""
    rng = np.random.default_rng(7)
    n, d, scale = 19, 8, 0.3
    q, k, v = (_rand(rng, n, d) for _ in range(3))
    u = _rand(rng, d)
    o1, lse1 = A.forward_head(q, k, v, scale, causal)
    o2, lse2 = A.forward_head(q, k + u[None, :], v, scale, causal)
    np.testing.assert_allclose(o2, o1, atol=1e-13)
    np.testing.assert_allclose(lse2 - lse1, scale * (q @ u), atol=1e-12)


def test_key_permutation_non_causal():
    rng = np.random.default_rng(8)
    n, d = 21, 8
    q, k, v = (_rand(rng, n, d) for _ in range(3))
    perm = rng.permutation(n)
    o1, lse1 = A.forward_head(q, k, v, 0.3, False)
    o2, lse2 = A.forward_head(q, k[perm], v[perm], 0.3, False)
    np.testing.assert_allclose(o2, o1, atol=1e-14)
    np.testing.assert_allclose(lse2, lse1, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,d", [(1, 3), (3, 2), (4, 4), (8, 4)])
def test_finite_differences(causal, n, d):
    """Central differences of loss = sum(O * G) in float64 (h = 1e-6) against
    the analytic dQ, dK, dV with dO = G."""
    rng = np.random.default_rng(100 + n * 10 + d)
    scale = 0.45
    q, k, v, gmat = (_rand(rng, n, d) for _ in range(4))
    g = A.backward_head(q, k, v, gmat, scale, causal)

    def loss(qq, kk, vv):
        return float(np.sum(A.forward_head(qq, kk, vv, scale, causal)[0] * gmat))

    h = 1e-6
    for name, idx in (("dq", 0), ("dk", 1), ("dv", 2)):
        base = [q, k, v]
        num = np.zeros((n, d))
        for i in range(n):
            for c in range(d):
                plus = [x.copy() for x in base]
                minus = [x.copy() for x in base]
                plus[idx][i, c] += h
                minus[idx][i, c] -= h
                num[i, c] = (loss(*plus) - loss(*minus)) / (2 * h)
        ana = g[name]
        denom = max(1.0, float(np.max(np.abs(ana))))
        assert np.max(np.abs(num - ana)) / denom <= 1e-6, name


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,d", [(1, 2), (2, 3), (3, 1), (4, 4)])
def test_brute_force(causal, n, d):
    rng = np.random.default_rng(200 + n * 10 + d)
    q, k, v, do = (_rand(rng, n, d) for _ in range(4))
    scale = 0.6
    o, lse = A.forward_head(q, k, v, scale, causal)
    bo, blse = brute.forward_head(q.tolist(), k.tolist(), v.tolist(), scale, causal)
    np.testing.assert_allclose(o, np.array(bo), atol=1e-14)
    np.testing.assert_allclose(lse, np.array(blse), atol=1e-14)
    g = A.backward_head(q, k, v, do, scale, causal)
    bq, bk, bv = brute.backward_head(q.tolist(), k.tolist(), v.tolist(), do.tolist(),
                                     scale, causal)
    np.testing.assert_allclose(g["dq"], np.array(bq), atol=1e-14)
    np.testing.assert_allclose(g["dk"], np.array(bk), atol=1e-14)
    np.testing.assert_allclose(g["dv"], np.array(bv), atol=1e-14)


def test_batched_layout_matches_heads():
    """The [B, N, H, d] / [B, H, N] entry points slice heads correctly."""
    rng = np.random.default_rng(9)
    B, N, H, d = 2, 9, 3, 4
    q, k, v, do = (_rand(rng, B, N, H, d) for _ in range(4))
    o, lse = A.forward(q, k, v, 0.5, True)
    dq, dk, dv, dd = A.backward(q, k, v, do, 0.5, True)
    for b in range(B):
        for h in range(H):
            oh, lh = A.forward_head(q[b, :, h], k[b, :, h], v[b, :, h], 0.5, True)
            assert np.array_equal(o[b, :, h], oh) and np.array_equal(lse[b, h], lh)
            g = A.backward_head(q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h], 0.5, True)
            assert np.array_equal(dq[b, :, h], g["dq"]) and np.array_equal(dd[b, h], g["D"])
            assert np.array_equal(dk[b, :, h], g["dk"]) and np.array_equal(dv[b, :, h], g["dv"])


# ---------------------------------------------------------------------------
# Online softmax: worked examples printed on the pages
# ---------------------------------------------------------------------------

def test_vector_trace_matches_page(golden):
    g = golden("online_softmax_vector.json")
    x = g["values"]
    tr = OS.trace(x, tile=1)
    bt = OS.trace(x, tile=1, broken=True)
    for (m, l), want in zip(tr, g["trace"]):
        assert m == pytest.approx(want["m"], abs=5e-5)
        assert l == pytest.approx(want["l"], abs=5e-5)
    for (m, l), want in zip(bt, g["brokenTrace"]):
        assert m == pytest.approx(want["m"], abs=5e-5)
        assert l == pytest.approx(want["l"], abs=5e-5)
    assert tr[-1][1] == pytest.approx(g["sum"], abs=5e-5)
    assert bt[-1][1] == pytest.approx(g["brokenSum"], abs=5e-5)
    assert OS.max_rises(x) == g["maxRises"]
    diff = np.max(np.abs(OS.online_weights(x) - OS.two_pass_weights(x)))
    assert diff <= 4 * g["maxWeightDiff"]


def test_probe_traces_tiles_of_four(golden):
    """Scores printed to 4 decimals, so the trace matches to ~5e-4."""
    g = golden("probe_heads.json")
    for head in g["heads"]:
        row = np.array(head["row"])
        tr = OS.trace(row, tile=g["tile"])
        assert len(tr) == len(head["trace"])
        for (m, l), want in zip(tr, head["trace"]):
            assert m == pytest.approx(want["m"], abs=5e-4)
            assert l == pytest.approx(want["l"], abs=5e-4)
        assert float(row.max()) == pytest.approx(head["rowMax"], abs=1e-9)
        assert int(np.argmax(row)) == head["argmax"]
        # the oracle's LSE of the same row equals the final (m, l) of the page
        _, lse = A.forward_head(row[None, :], np.eye(row.size), np.eye(row.size),
                                1.0, False)
        m_f, l_f = head["trace"][-1]["m"], head["trace"][-1]["l"]
        assert lse[0] == pytest.approx(m_f + math.log(l_f), abs=5e-4)


def test_film_table_rows_and_sweep(golden):
    """The causal score table of the largest-score head: its last row is the
    probe row (3 vs 4 decimals), and each row's tiles-of-4 trace through the
    oracle's (m, l) merge agrees with the oracle's LSE."""
    g = golden("film_table.json")
    probe = golden("probe_heads.json")
    rows = g["scores"]
    n = len(rows)
    ph = [h for h in probe["heads"] if h["layer"] == g["layer"] and h["head"] == g["head"]][0]
    np.testing.assert_allclose(rows[-1], ph["row"], atol=6e-4)
    # the whole table as a causal score matrix: q = scores (padded), k = I
    s = np.zeros((n, n))
    for i, r in enumerate(rows):
        assert len(r) == i + 1
        s[i, :i + 1] = r
    _, lse = A.forward_head(s, np.eye(n), np.eye(n), 1.0, True)
    for i, r in enumerate(rows):
        st = (-np.inf, 0.0)
        for t0 in range(0, len(r), 4):
            blk = np.array(r[t0:t0 + 4])
            st = OS.merge(st, (float(blk.max()), float(np.exp(blk - blk.max()).sum())))
        assert lse[i] == pytest.approx(st[0] + math.log(st[1]), abs=1e-12)
    for head in g["sweep"]["heads"]:
        want = [h for h in probe["heads"]
                if h["layer"] == head["layer"] and h["head"] == head["head"]][0]
        assert head["trace"] == want["trace"]
        rises = sum(1 for a, b in zip(head["trace"], head["trace"][1:]) if b["m"] > a["m"])
        assert rises == head["rises"]


def test_online_merge_associative_and_equal_to_two_pass():
    rng = np.random.default_rng(10)
    for trial in range(50):
        x = rng.normal(0, 3, size=int(rng.integers(1, 60)))
        # random split points, random bracketing
        cuts = sorted(set(rng.integers(0, x.size, size=int(rng.integers(0, 6))).tolist()))
        parts = [p for p in np.split(x, cuts) if p.size]
        states = [(float(p.max()), float(np.exp(p - p.max()).sum())) for p in parts]
        while len(states) > 1:
            i = int(rng.integers(0, len(states) - 1))
            states[i:i + 2] = [OS.merge(states[i], states[i + 1])]
        m, l = states[0]
        assert m == x.max()
        assert l == pytest.approx(np.exp(x - x.max()).sum(), rel=1e-13)
        # commutative
        a, b = (1.5, 2.0), (-0.5, 3.0)
        assert OS.merge(a, b) == pytest.approx(OS.merge(b, a), rel=1e-15)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n", [1, 7, 20, 33])
def test_tiled_restatement_equals_oracle(causal, n):
    rng = np.random.default_rng(11 + n)
    d = 5
    q, k, v = (_rand(rng, n, d, sigma=2.0) for _ in range(3))
    o, lse = A.forward_head(q, k, v, 0.5, causal)
    for br, bc in [(1, 1), (4, 3), (16, 16), (n, n), (5, 64)]:
        to, tl, _ = OS.tiled_attention_head(q, k, v, 0.5, causal, br, bc)
        np.testing.assert_allclose(to, o, atol=1e-13)
        np.testing.assert_allclose(tl, lse, atol=1e-13)


def test_broken_rescale_fails_only_when_rows_span_tiles():
    rng = np.random.default_rng(12)
    n, d = 48, 8
    q, k, v = (_rand(rng, n, d, sigma=2.0) for _ in range(3))
    o, _ = A.forward_head(q, k, v, 0.5, False)
    one_tile, _, _ = OS.tiled_attention_head(q, k, v, 0.5, False, 16, n, broken=True)
    assert checker.mismatches(one_tile, o, 1e-12) == 0
    many, _, _ = OS.tiled_attention_head(q, k, v, 0.5, False, 16, 8, broken=True)
    assert checker.mismatches(many, o, 1e-3) > 0


# ---------------------------------------------------------------------------
# Checker self-test (mirrors the facts page's controls.checker)
# ---------------------------------------------------------------------------

def test_checker_controls():
    rng = np.random.default_rng(13)
    n, d = 256, 16
    q, k, v = (_rand(rng, n, d) for _ in range(3))
    o, _ = A.forward_head(q, k, v, 0.25, False)
    tiled32, _, _ = OS.tiled_attention_head(q, k, v, 0.25, False, 128, 16,
                                            dtype=np.float32)
    assert checker.mismatches(tiled32, o, 1e-5) == 0          # tiled float32 passes
    rounded = o.astype(np.float32)
    assert checker.mismatches(rounded, o, 1e-5) == 0          # exact, rounded, passes
    moved = rounded.astype(np.float64).copy()
    moved[77, 3] += 1e-3
    assert checker.mismatches(moved, o, 1e-5) == 1            # exactly one mismatch
    assert checker.mismatches(tiled32, o, 0.0) > 0            # zero tolerance rejects
    bad = rounded.astype(np.float64).copy()
    bad[5, 5] = np.nan
    assert checker.mismatches(bad, o, 1.0) == 1               # NaN is a mismatch


def test_float32_restatement_error_magnitude(golden):
    """A float32 restatement of the fused loop on uniform[-2, 2) inputs lands in
    the error range the page reports for its float32 emulation (max-abs errors
    of 3.4e-7 .. 8.3e-7 for the fused kernel); the broken one is far off."""
    g = golden("correctness.json")
    rng = np.random.default_rng(1)
    for row in g["rows"]:
        if row["N"] != 256 or row["kind"] == "unfused":
            continue
        n, d, tile = row["N"], row["d"], row["B"]
        q, k, v = (rng.uniform(-2, 2, size=(n, d)) for _ in range(3))
        q, k, v = (x.astype(np.float32).astype(np.float64) for x in (q, k, v))
        scale = 1.0 / math.sqrt(d)
        o, _ = A.forward_head(q, k, v, scale, False)
        out, _, _ = OS.tiled_attention_head(q, k, v, scale, False, tile, tile,
                                            broken=(row["kind"] == "broken"),
                                            dtype=np.float32)
        err = checker.max_abs_err(out, o)
        if row["ok"]:
            assert row["maxErr"] / 20 <= err <= row["maxErr"] * 20
        else:
            assert row["maxErr"] / 10 <= err <= row["maxErr"] * 10


# ---------------------------------------------------------------------------
# fp16 overflow numbers and traffic closed forms
# ---------------------------------------------------------------------------

def test_fp16_overflow_pins(golden):
    g = golden("overflow.json")
    probe = golden("probe_heads.json")
    assert fp16_softmax.FP16_OVERFLOW_THRESHOLD == pytest.approx(g["threshold"], abs=5e-5)
    assert np.isinf(np.float16(np.exp(g["threshold"] + 1e-4)))
    assert np.isfinite(np.float16(np.exp(g["threshold"] - 1e-4)))
    pr = g["probeRow"]
    row = [h for h in probe["heads"] if h["layer"] == pr["layer"] and h["head"] == pr["head"]][0]["row"]
    w, s = fp16_softmax.naive_fp16(row)
    assert float(np.float16(np.exp(pr["max"]))) == pr["expOfMax"]
    assert float(s) == pr["naiveSum"] and np.isfinite(s)
    ws, ss = fp16_softmax.safe_fp16(row)
    assert float(ss) == pytest.approx(pr["safeSum"], abs=1e-3)
    assert fp16_softmax.overflow_factor(row) == pytest.approx(pr["overflowFactor"], abs=5e-5)


def test_traffic_closed_forms(golden):
    g = golden("traffic.json")
    assert len(g["rows"]) == 28
    for row in g["rows"]:
        c = traffic.counts(row["N"], row["d"], row["B"], row["kind"])
        for key in ("globalReads", "globalWrites", "globalBytes", "extraMemoryBytes",
                    "fma", "exps"):
            assert c[key] == row[key], (row, key)
