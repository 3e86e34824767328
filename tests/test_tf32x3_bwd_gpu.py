"""float32 backward on the tensor cores (fa_bwd_tf32x3, 3xTF32) against the
float64 oracle's analytic gradients at the float32 gradient tolerance (1e-4),
and against the float32 FMA path's gradients."""

import os

import pytest

from exact_attention_fwd_gb300.configs import WORKLOADS
from tests.gpu_util import TOL, default_scale, make, require_gpu
from tests.test_bwd_gpu import compare_bwd

pytestmark = pytest.mark.gpu


def _run(inp, causal, scale):
    """The forward on the FMA path, then fa_bwd_tf32x3; every output row is
    pre-filled with NaN so a row the kernels never write fails the check."""
    import torch
    from exact_attention_fwd_gb300 import api
    dev = torch.device("cuda", 0)
    q, k, v, do = (inp.torch(t, dev) for t in ("q", "k", "v", "do"))
    o, lse = api.forward(q, k, v, scale=scale, causal=causal)
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    api.backward_tf32x3(q, k, v, o, lse, do, scale=scale, causal=causal, dq=dq, dk=dk, dv=dv)
    assert api.sync_status() == 0
    return dict(q=q, k=k, v=v, do=do, o=o, lse=lse, dq=dq, dk=dk, dv=dv)


@pytest.mark.parametrize("sub", range(5))
def test_causal_sweep_backward_tf32x3(sub):
    """Workload 1's causal shapes (the float32 parity sweep)."""
    require_gpu()
    w = WORKLOADS[1]
    s = w.shapes[sub]
    inp = make(s.B, s.H, s.N, s.d, "f32", w.seed(sub))
    out = _run(inp, True, w.scale(s))
    compare_bwd(inp, out, True, w.scale(s), TOL["f32"]["grad"])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,d", [
    (1, 1, 64, 16), (2, 2, 300, 64), (1, 3, 129, 32), (1, 2, 1, 8), (2, 1, 257, 40),
    (1, 2, 33, 24), (1, 2, 640, 64),
])
def test_shapes_backward_tf32x3(B, H, N, d, causal):
    """Several 128-row tiles, ragged tails (N not a multiple of the 32-row
    blocks or the 128-row tiles), head dims below the padded 64, one key."""
    require_gpu()
    inp = make(B, H, N, d, "f32", 17000 + N + d)
    out = _run(inp, causal, default_scale(d))
    compare_bwd(inp, out, causal, default_scale(d), TOL["f32"]["grad"])


@pytest.mark.parametrize("scale", [0.0, -0.25])
def test_unusual_scales_backward_tf32x3(scale):
    require_gpu()
    inp = make(1, 2, 200, 64, "f32", 17100)
    for causal in (False, True):
        out = _run(inp, causal, scale)
        compare_bwd(inp, out, causal, scale, TOL["f32"]["grad"])


def test_matches_fma_path():
    """Against fa_bwd's float32 FMA path on the same inputs: two float32
    computations of the same gradients, each within 1e-4 of the float64
    oracle, agree within that bar too (measured: 3.2e-5 on dV here, the
    float32 summation orders differ)."""
    torch = require_gpu()
    from exact_attention_fwd_gb300 import api
    inp = make(2, 2, 384, 64, "f32", 17200)
    out = _run(inp, True, default_scale(64))
    ref = api.backward(out["q"], out["k"], out["v"], out["o"], out["lse"], out["do"],
                       scale=default_scale(64), causal=True)
    assert api.sync_status() == 0
    for name, r in zip(("dq", "dk", "dv"), ref):
        err = float((out[name] - r).abs().max())
        assert err <= TOL["f32"]["grad"], f"{name}: {err:.3e}"


def test_unsupported_head_dim_tf32x3():
    torch = require_gpu()
    from exact_attention_fwd_gb300 import _lib, api
    inp = make(1, 1, 64, 128, "f32", 17300)
    dev = torch.device("cuda", 0)
    q, k, v, do = (inp.torch(t, dev) for t in ("q", "k", "v", "do"))
    o, lse = api.forward(q, k, v, causal=True)
    with pytest.raises(_lib.FaError) as e:
        api.backward_tf32x3(q, k, v, o, lse, do, causal=True)
    assert e.value.status == _lib.FA_ERR_UNSUPPORTED
    assert api.sync_status() == 0


def test_backward_tf32x3_bounded_wait_self_test():
    """The self-test switch makes each kernel's first wait time out:
    FA_ERR_TIMEOUT through the status word, the context stays usable."""
    torch = require_gpu()
    from exact_attention_fwd_gb300 import _lib, api
    inp = make(1, 2, 256, 64, "f32", 17400)
    dev = torch.device("cuda", 0)
    q, k, v, do = (inp.torch(t, dev) for t in ("q", "k", "v", "do"))
    o, lse = api.forward(q, k, v, causal=True)
    assert api.sync_status() == 0
    os.environ["FA_SELFTEST_WAIT_TIMEOUT"] = "1"
    try:
        api.backward_tf32x3(q, k, v, o, lse, do, causal=True)
        st = api.sync_status()
    finally:
        del os.environ["FA_SELFTEST_WAIT_TIMEOUT"]
    assert st == _lib.FA_ERR_TIMEOUT
    assert api.sync_status() == 0
    out = _run(inp, True, default_scale(64))
    compare_bwd(inp, out, True, default_scale(64), TOL["f32"]["grad"])
