"""fa_fwd_bwd_host (host buffers, chunked copy/compute pipeline) on the GPU:
its results equal the device-buffer calls bit for bit (each head's arithmetic
does not depend on the batch it is computed in), and match the oracle."""

import numpy as np
import pytest

from exact_attention_fwd_gb300.inputs import torch_to_f64
from tests.gpu_util import TOL, compare_fwd, default_scale, make, require_gpu
from tests.test_bwd_gpu import compare_bwd

pytestmark = pytest.mark.gpu


def _host(inp, t, pin=True):
    x = inp.torch(t, "cpu")
    return x.pin_memory() if pin else x


@pytest.mark.parametrize("B,chunk", [(5, 2), (4, 4), (3, 8), (6, 1), (13, 4)])
@pytest.mark.parametrize("causal", [False, True])
def test_host_equals_device_calls(B, chunk, causal):
    torch = require_gpu()
    from exact_attention_fwd_gb300 import api
    inp = make(B, 2, 300, 64, "bf16", 14000 + B * 10 + chunk)
    qh, kh, vh, doh = (_host(inp, t) for t in ("q", "k", "v", "do"))
    o, lse, dq, dk, dv = api.fwd_bwd_host(qh, kh, vh, doh, chunk, causal=causal)
    torch.cuda.synchronize()
    assert api.sync_status() == 0
    dev = torch.device("cuda", 0)
    q, k, v, do = (t.to(dev) for t in (qh, kh, vh, doh))
    o_d, l_d = api.forward(q, k, v, causal=causal)
    g = api.backward(q, k, v, o_d, l_d, do, causal=causal)
    assert api.sync_status() == 0
    for a, b in ((o, o_d), (lse, l_d), (dq, g[0]), (dk, g[1]), (dv, g[2])):
        assert torch.equal(a, b.cpu())


def test_host_matches_oracle_fp32_grads_pageable():
    """Pageable host buffers (no overlap, same results), fp32 gradients."""
    torch = require_gpu()
    from exact_attention_fwd_gb300 import api
    inp = make(3, 2, 200, 64, "bf16", 14100)
    qh, kh, vh, doh = (_host(inp, t, pin=False) for t in ("q", "k", "v", "do"))
    o, lse, dq, dk, dv = api.fwd_bwd_host(qh, kh, vh, doh, 2, causal=True,
                                          grad_dtype=torch.float32)
    torch.cuda.synchronize()
    assert api.sync_status() == 0
    compare_fwd(inp, o, lse, True, default_scale(64))
    compare_bwd(inp, {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}, True, default_scale(64),
                TOL["bf16"]["grad"])
