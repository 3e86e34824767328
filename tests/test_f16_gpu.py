"""fp16 I/O (FA_DTYPE_F16) on the GPU: the same tcgen05 kernels with fp16
storage, against the float64 oracle on the same fp16-rounded inputs."""

import pytest

from exact_attention_fwd_gb300.configs import WORKLOADS
from tests.gpu_util import TOL, compare_fwd, default_scale, make, require_gpu, run_fwd
from tests.test_bwd_gpu import compare_bwd, run_fwd_bwd

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("sub", range(5))
def test_causal_sweep_f16(sub):
    """Workload 1's causal shapes with fp16 storage, forward and backward."""
    require_gpu()
    w = WORKLOADS[1]
    s = w.shapes[sub]
    inp = make(s.B, s.H, s.N, s.d, "f16", w.seed(sub))
    out = run_fwd_bwd(inp, causal=True)
    compare_fwd(inp, out["o"], out["lse"], True, w.scale(s))
    compare_bwd(inp, out, True, w.scale(s), TOL["f16"]["grad"])


@pytest.mark.parametrize("d", [8, 40, 64, 96, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_head_dims_f16(d, causal):
    require_gpu()
    inp = make(2, 2, 300, d, "f16", 11000 + d)
    out = run_fwd_bwd(inp, causal=causal)
    compare_fwd(inp, out["o"], out["lse"], causal, default_scale(d))
    compare_bwd(inp, out, causal, default_scale(d), TOL["f16"]["grad"])


@pytest.mark.parametrize("N", [1, 127, 129, 640])
def test_ragged_n_f16(N):
    require_gpu()
    inp = make(1, 2, N, 64, "f16", 11500 + N)
    for causal in (False, True):
        out = run_fwd_bwd(inp, causal=causal)
        compare_fwd(inp, out["o"], out["lse"], causal, default_scale(64))
        compare_bwd(inp, out, causal, default_scale(64), TOL["f16"]["grad"])


def test_large_scores_f16_fp32_gradients():
    """Q, K ~ N(0, 4^2): large score ranges, rescaling; float32 gradients."""
    require_gpu()
    inp = make(2, 4, 512, 64, "f16", 11900, sigma={"q": 4.0, "k": 4.0})
    for causal in (False, True):
        out = run_fwd_bwd(inp, causal=causal, grad_f32=True)
        compare_fwd(inp, out["o"], out["lse"], causal, default_scale(64))
        compare_bwd(inp, out, causal, default_scale(64), TOL["f16"]["grad"])


@pytest.mark.parametrize("scale", [0.0, -0.3])
def test_unusual_scales_f16(scale):
    require_gpu()
    inp = make(1, 2, 300, 64, "f16", 12000)
    for causal in (False, True):
        o, lse, _ = run_fwd(inp, causal=causal, scale=scale)
        compare_fwd(inp, o, lse, causal, scale)


def test_causal_first_row_equals_v0_f16():
    torch = require_gpu()
    inp = make(2, 3, 300, 64, "f16", 12100)
    o, lse, (q, k, v) = run_fwd(inp, causal=True)
    assert o.dtype == torch.float16
    assert torch.equal(o[:, 0], v[:, 0])


def test_scores_beyond_fp16_exp_range():
    """Scaled scores up to ~30, past ln 65520 = 11.09 where a naive fp16
    exponential overflows (the facts page's "overflow" entry): the kernel
    subtracts the running max in fp32 before exponentiating, so O and L stay
    finite and match the oracle."""
    torch = require_gpu()
    inp = make(1, 2, 192, 64, "f16", 12200)
    for causal in (False, True):
        o, lse, _ = run_fwd(inp, causal=causal, scale=1.0)
        assert torch.isfinite(o).all() and torch.isfinite(lse).all()
        assert float(lse.max()) > 11.0901
        compare_fwd(inp, o, lse, causal, 1.0)
