"""Forward parity on the GPU: the CUDA path through the C ABI against the
float64 oracle, element by element, on seeded inputs."""

import os

import numpy as np
import pytest

from exact_attention_fwd_gb300.configs import BROWSER_SHAPE, WORKLOADS
from tests.gpu_util import (TOL, compare_fwd, default_scale, make, require_gpu, run_fwd)

pytestmark = pytest.mark.gpu


def test_single_head_f32():
    """Workload 0: B1 H1 N64 d16 fp32, no mask."""
    require_gpu()
    w = WORKLOADS[0]
    s = w.shapes[0]
    inp = make(s.B, s.H, s.N, s.d, "f32", w.seed(0))
    o, lse, _ = run_fwd(inp, causal=False)
    eo, el = compare_fwd(inp, o, lse, False, w.scale(s))
    assert eo < TOL["f32"]["o"] and el < TOL["f32"]["lse"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("sub", range(5))
def test_causal_sweep(dtype, sub):
    """Workload 1: the pages' causal parity shapes, fp32 and bf16."""
    require_gpu()
    w = WORKLOADS[1]
    s = w.shapes[sub]
    inp = make(s.B, s.H, s.N, s.d, dtype, w.seed(sub))
    o, lse, _ = run_fwd(inp, causal=True)
    compare_fwd(inp, o, lse, True, w.scale(s))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_browser_shape(dtype, causal):
    require_gpu()
    s = BROWSER_SHAPE
    inp = make(s.B, s.H, s.N, s.d, dtype, 5000 + int(causal))
    o, lse, _ = run_fwd(inp, causal=causal)
    compare_fwd(inp, o, lse, causal, default_scale(s.d))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 2, 127, 128, 129, 255, 256, 257, 300, 385, 640])
def test_ragged_n_bf16(causal, N):
    """Several 128-row tiles, 256-row tile pairs, and ragged tails."""
    require_gpu()
    inp = make(1, 2, N, 64, "bf16", 6000 + N)
    o, lse, _ = run_fwd(inp, causal=causal)
    compare_fwd(inp, o, lse, causal, default_scale(64))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [160, 193, 224, 287])
def test_row_quarter_boundaries_bf16(causal, N):
    """Sequence ends inside each 32-row quarter of a 128-row tile: each warp
    stores its own 32 output rows (a box partly or wholly past N), and the
    keep masks of the ragged and diagonal blocks end inside a 32-column word.
    Several heads, so that CTAs run more than one item."""
    require_gpu()
    inp = make(2, 5, N, 64, "bf16", 6500 + N)
    o, lse, _ = run_fwd(inp, causal=causal)
    compare_fwd(inp, o, lse, causal, default_scale(64))


@pytest.mark.parametrize("d", [8, 16, 24, 32, 40, 56, 64, 72, 96, 120, 128])
def test_head_dims_bf16(d):
    require_gpu()
    inp = make(2, 2, 200, d, "bf16", 7000 + d)
    for causal in (False, True):
        o, lse, _ = run_fwd(inp, causal=causal)
        compare_fwd(inp, o, lse, causal, default_scale(d))


@pytest.mark.parametrize("d", [8, 24, 64, 128])
def test_head_dims_f32(d):
    require_gpu()
    inp = make(1, 3, 77, d, "f32", 7500 + d)
    for causal in (False, True):
        o, lse, _ = run_fwd(inp, causal=causal)
        compare_fwd(inp, o, lse, causal, default_scale(d))


def test_large_scores_bf16():
    """Q, K ~ N(0, 4^2) as in the BERT-shaped workload: large score ranges make
    the running max rise and exercise the rescale."""
    require_gpu()
    inp = make(2, 2, 700, 64, "bf16", 8000, sigma={"q": 4.0, "k": 4.0})
    for causal in (False, True):
        o, lse, _ = run_fwd(inp, causal=causal)
        compare_fwd(inp, o, lse, causal, default_scale(64))


@pytest.mark.parametrize("scale", [0.0, -0.3, 2.0])
def test_unusual_scales_bf16(scale):
    require_gpu()
    inp = make(1, 2, 300, 64, "bf16", 8100)
    for causal in (False, True):
        o, lse, _ = run_fwd(inp, causal=causal, scale=scale)
        compare_fwd(inp, o, lse, causal, scale)


def test_causal_first_row_equals_v0():
    """Row 0 of a causal forward sees only key 0, so O[0] = V[0] (bf16 exact)."""
    torch = require_gpu()
    inp = make(2, 3, 300, 64, "bf16", 8200)
    o, lse, (q, k, v) = run_fwd(inp, causal=True)
    assert torch.equal(o[:, 0], v[:, 0])


def test_repeat_is_bitwise_deterministic():
    torch = require_gpu()
    inp = make(2, 2, 513, 128, "bf16", 8300)
    o1, l1, _ = run_fwd(inp, causal=True)
    o2, l2, _ = run_fwd(inp, causal=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_guard_bands_untouched():
    """Outputs written through views into larger buffers: the bytes around them
    keep their fill pattern."""
    torch = require_gpu()
    from exact_attention_fwd_gb300 import api
    inp = make(1, 2, 200, 64, "bf16", 8400)
    dev = torch.device("cuda", 0)
    q, k, v = (inp.torch(t, dev) for t in ("q", "k", "v"))
    pad = 4096
    n_o, n_l = q.numel(), 2 * 200
    o_buf = torch.full((n_o + 2 * pad,), 7.0, dtype=torch.bfloat16, device=dev)
    l_buf = torch.full((n_l + 2 * pad,), 7.0, dtype=torch.float32, device=dev)
    o = o_buf[pad:pad + n_o].view(q.shape)
    lse = l_buf[pad:pad + n_l].view(1, 2, 200)
    api.forward(q, k, v, causal=True, out=o, lse=lse)
    assert api.sync_status() == 0
    assert torch.all(o_buf[:pad] == 7.0) and torch.all(o_buf[pad + n_o:] == 7.0)
    assert torch.all(l_buf[:pad] == 7.0) and torch.all(l_buf[pad + n_l:] == 7.0)
    compare_fwd(inp, o, lse, True, default_scale(64))


def test_bounded_wait_self_test_reports_timeout():
    """With the self-test switch set, the kernel's first wait is on a barrier
    nothing arrives on: it must give up, report FA_ERR_TIMEOUT through the
    status word and leave the context usable."""
    torch = require_gpu()
    from exact_attention_fwd_gb300 import _lib, api
    inp = make(1, 2, 256, 64, "bf16", 8500)
    dev = torch.device("cuda", 0)
    q, k, v = (inp.torch(t, dev) for t in ("q", "k", "v"))
    os.environ["FA_SELFTEST_WAIT_TIMEOUT"] = "1"
    try:
        api.forward(q, k, v, causal=True)
        st = api.sync_status()
    finally:
        del os.environ["FA_SELFTEST_WAIT_TIMEOUT"]
    assert st == _lib.FA_ERR_TIMEOUT
    assert api.sync_status() == 0          # cleared
    o, lse = api.forward(q, k, v, causal=True)
    assert api.sync_status() == 0
    compare_fwd(inp, o, lse, True, default_scale(64))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(200, 64), (300, 64), (650, 128)])
def test_many_items_per_cta(causal, N, d):
    """Enough (b, h) heads that every persistent CTA walks several work items,
    including single-tile items (odd tile counts); sampled heads in full."""
    require_gpu()
    B, H = 40, 16
    inp = make(B, H, N, d, "bf16", 8600 + N + int(causal))
    o, lse, _ = run_fwd(inp, causal=causal)
    heads = [(0, 0), (B - 1, H - 1), (17, 5), (23, 11), (39, 0)]
    compare_fwd(inp, o, lse, causal, default_scale(d), heads=heads)


def test_status_word_is_shared_across_streams():
    """The device status word is one per device: a timeout recorded by a
    kernel on stream A is what fa_sync_status on stream B reports, and that
    call clears it for A as well (documented in include/fa.h)."""
    torch = require_gpu()
    from exact_attention_fwd_gb300 import _lib, api
    inp = make(1, 2, 256, 64, "bf16", 8801)
    dev = torch.device("cuda", 0)
    q, k, v = (inp.torch(t, dev) for t in ("q", "k", "v"))
    sa, sb = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    torch.cuda.synchronize(dev)
    assert api.sync_status() == 0
    os.environ["FA_SELFTEST_WAIT_TIMEOUT"] = "1"
    try:
        api.forward(q, k, v, causal=True, stream=sa)
    finally:
        del os.environ["FA_SELFTEST_WAIT_TIMEOUT"]
    sa.synchronize()                              # the kernel on A has finished
    assert api.sync_status(stream=sb) == _lib.FA_ERR_TIMEOUT
    assert api.sync_status(stream=sa) == 0        # already read and cleared via B
    o, lse = api.forward(q, k, v, causal=True, stream=sb)
    assert api.sync_status(stream=sb) == 0
    compare_fwd(inp, o, lse, True, default_scale(64))
