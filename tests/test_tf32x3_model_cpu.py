"""The 3xTF32 error model behind the float32 tensor-core forward's tolerances (CPU).

Each float32 x is split as hi = tf32(x), lo = tf32(x - hi) (nearest tf32
value, ties away from zero), and a product x y is taken as
hi_x hi_y + hi_x lo_y + lo_x hi_y.  These tests pin each step of the bound
the GPU test's tolerances are derived from, on a numpy model of the split
(float64 accumulation, so only the split's own error is measured), against
the float64 oracle:

* tf32 rounding moves x by at most 2^-11 |x| and leaves 13 zero low bits;
* x - hi is exact in float32, so lo carries the whole remainder up to its own
  rounding: |x - hi - lo| <= 2^-22 |x|;
* the three-product form misses x y by at most about 3 * 2^-22 |x y|;
* through attention the model stays inside the bars the GPU test uses:
  float32 (O 1e-5, L 1e-4) at sigma = 1, and O 5e-5, L 2e-4 at sigma = 4
  (measured here: at most 2.4e-7 and 4.8e-6), so the split is not what limits
  the GPU result, and a single tf32 product (hi only) misses the float32 bar
  by more than an order of magnitude.
"""
import numpy as np
import pytest

from exact_attention_fwd_gb300.inputs import Inputs
from oracle import attention as oracle

F32 = np.float32


def tf32(x):
    """Nearest tf32 value of float32 `x` (ties away from zero), as float32."""
    b = np.ascontiguousarray(x, dtype=F32).view(np.uint32)
    return ((b + np.uint32(0x1000)) & np.uint32(0xFFFFE000)).view(F32)


def split(x):
    x = np.asarray(x, dtype=F32)
    hi = tf32(x)
    lo = tf32(x - hi)
    return hi, lo


def _normals(n, seed=7, scale=1.0):
    rng = np.random.default_rng(seed)
    return (rng.normal(0.0, scale, n) * np.exp(rng.uniform(-20, 20, n))).astype(F32)


def test_tf32_rounding_bound_and_format():
    x = _normals(200000)
    t = tf32(x)
    assert np.all((t.view(np.uint32) & np.uint32(0x1FFF)) == 0)
    x64, t64 = x.astype(np.float64), t.astype(np.float64)
    assert np.all(np.abs(x64 - t64) <= 2.0 ** -11 * np.abs(x64))
    # nearest: no other tf32 neighbour is closer
    ulp = np.ldexp(1.0, np.frexp(t64)[1] - 11)     # spacing of tf32 values at t
    assert np.all(np.abs(x64 - t64) <= 0.5 * ulp * (1 + 1e-12))


def test_split_remainder_is_exact_and_small():
    x = _normals(200000, seed=8)
    hi, lo = split(x)
    x64, hi64, lo64 = (a.astype(np.float64) for a in (x, hi, lo))
    # x - hi is exact in float32
    assert np.array_equal((x - hi).astype(np.float64), x64 - hi64)
    assert np.all(np.abs(x64 - hi64 - lo64) <= 2.0 ** -22 * np.abs(x64))


def test_three_product_error_bound():
    x, y = _normals(200000, seed=9), _normals(200000, seed=10)
    hx, lx = split(x)
    hy, ly = split(y)
    exact = x.astype(np.float64) * y.astype(np.float64)
    approx = (hx.astype(np.float64) * hy + hx.astype(np.float64) * ly
              + lx.astype(np.float64) * hy)
    rel = np.abs(exact - approx) / np.abs(exact)
    assert rel.max() <= 3.01 * 2.0 ** -22
    # the dropped lo*lo term is the leading part: the bound is not loose by orders
    assert rel.max() > 2.0 ** -24


def _model_forward(q, k, v, scale, causal):
    """3xTF32 attention for one head in the model: split products, float64 sums."""
    f = np.float64
    qh, ql = (a.astype(f) for a in split(q))
    kh, kl = (a.astype(f) for a in split(k))
    vh, vl = (a.astype(f) for a in split(v))
    s = (qh @ kh.T + qh @ kl.T + ql @ kh.T) * scale
    n = s.shape[0]
    if causal:
        s[np.triu_indices(n, 1)] = -np.inf
    m = s.max(axis=1)
    p = np.exp(s - m[:, None]).astype(F32)          # P is a float32 value on the GPU
    ph, pl = (a.astype(f) for a in split(p))
    l = p.astype(f).sum(axis=1)
    o = (ph @ vh + ph @ vl + pl @ vh) / l[:, None]
    return o, m + np.log(l)


@pytest.mark.parametrize("sigma,tol_o,tol_l", [(1.0, 1e-5, 1e-4), (4.0, 5e-5, 2e-4)])
@pytest.mark.parametrize("causal", [False, True])
def test_model_attention_within_the_gpu_bars(sigma, tol_o, tol_l, causal):
    inp = Inputs(1, 1, 512, 64, "f32", 16500, sigma={"q": sigma, "k": sigma})
    q, k, v = (inp.storage[t][0, :, 0, :] for t in ("q", "k", "v"))
    scale = 1.0 / np.sqrt(64.0)
    o, lse = _model_forward(q, k, v, scale, causal)
    o_ref, lse_ref = oracle.forward_head(q.astype(np.float64), k.astype(np.float64),
                                         v.astype(np.float64), scale, causal)
    e_o = np.abs(o - o_ref).max()
    e_l = np.abs(lse - lse_ref).max()
    # the split's own error uses at most half of each bar; float32 accumulation
    # on the GPU takes the rest
    assert e_o <= 0.5 * tol_o, e_o
    assert e_l <= 0.5 * tol_l, e_l


def test_one_product_misses_the_float32_bar():
    """hi_x hi_y alone (plain TF32) cannot meet O 1e-5: the lo terms are needed."""
    inp = Inputs(1, 1, 512, 64, "f32", 16500)
    q, k, v = (inp.storage[t][0, :, 0, :] for t in ("q", "k", "v"))
    scale = 1.0 / np.sqrt(64.0)
    f = np.float64
    qh, kh, vh = (split(a)[0].astype(f) for a in (q, k, v))
    s = (qh @ kh.T) * scale
    m = s.max(axis=1)
    p = np.exp(s - m[:, None]).astype(F32)
    l = p.astype(f).sum(axis=1)
    o = (split(p)[0].astype(f) @ vh) / l[:, None]
    o_ref, _ = oracle.forward_head(q.astype(f), k.astype(f), v.astype(f), scale, False)
    assert np.abs(o - o_ref).max() > 10 * 1e-5
