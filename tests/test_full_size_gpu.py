"""Parity at the three full-size workloads, in the launch configuration the
benchmark times.

GPT-2-medium and BERT-large shapes: every row of every (b, h) head of O, LSE,
dQ, dK and dV against the float64 oracle (1024 heads each).  Long context
(N = 8192, d = 128): every row of 16 heads spread over all batch entries and
over both ends of each, i.e. over early and late, even and odd waves of the
persistent schedule (the oracle's N x N float64 matrices cost ~0.5 GB and
tens of seconds per head there).  The oracle runs in spawned host processes
(tests/fullsize_oracle.py).  Properties that hold on every head are checked
on all of them as well.
"""

import numpy as np
import pytest

from exact_attention_fwd_gb300.configs import WORKLOADS
from exact_attention_fwd_gb300.inputs import Inputs
from tests.fullsize_oracle import check_heads, workers_for
from tests.gpu_util import TOL, require_gpu

pytestmark = pytest.mark.gpu


def _run(w, grad_dtypes):
    torch = require_gpu()
    from exact_attention_fwd_gb300 import api
    s = w.shapes[0]
    inp = Inputs(s.B, s.H, s.N, s.d, "bf16", w.seed(0), w.sigma)
    dev = torch.device("cuda", 0)
    q, k, v, do = (inp.torch(t, dev) for t in ("q", "k", "v", "do"))
    scale = w.scale(s)
    o, lse = api.forward(q, k, v, scale=scale, causal=w.causal)
    out = dict(q=q, k=k, v=v, do=do, o=o, lse=lse)
    for tag, gdt in grad_dtypes.items():
        dq, dk, dv = api.backward(q, k, v, o, lse, do, scale=scale, causal=w.causal,
                                  grad_dtype=gdt)
        out.update({"dq" + tag: dq, "dk" + tag: dk, "dv" + tag: dv})
    assert api.sync_status() == 0
    return inp, scale, out


def _host(t):
    import torch
    if t.dtype == torch.bfloat16:
        return t.detach().view(torch.int16).cpu().numpy().view(np.uint16), "bf16"
    return t.detach().float().cpu().numpy(), "f32"


def _check_properties(w, out, tag=""):
    """On every head: with a causal mask row 0 of O equals V[0] exactly; the
    keys' dK sum to zero and the keys' dV sum to the queries' dO sum."""
    import torch
    if w.causal:
        assert torch.equal(out["o"][:, 0], out["v"][:, 0])
    dk_sum = out["dk" + tag].float().sum(dim=1)
    assert float(dk_sum.abs().max()) < 1.0
    dv_sum = out["dv" + tag].float().sum(dim=1)
    do_sum = out["do"].float().sum(dim=1)
    assert float((dv_sum - do_sum).abs().max()) < 1.0
    for t in ("o", "lse", "dq" + tag, "dk" + tag, "dv" + tag):
        assert bool(torch.isfinite(out[t]).all()), t


def _all_heads(inp):
    return [(b, h) for b in range(inp.B) for h in range(inp.H)]


def _assert_clean(worst, fails, what):
    print(f"\n{what}: worst max-abs errors {dict(sorted(worst.items()))}")
    assert not fails, f"{len(fails)} failures, first: {fails[:5]}"


def test_gpt2_medium_shape_full_size():
    w = WORKLOADS[2]
    inp, scale, out = _run(w, {"": None})
    _check_properties(w, out)
    outputs = {n: _host(out[n]) for n in ("o", "lse", "dq", "dk", "dv")}
    worst, fails = check_heads(inp, outputs, _all_heads(inp), scale, w.causal, TOL["bf16"])
    _assert_clean(worst, fails, "GPT-2 shape, all 1024 heads")


def test_bert_large_shape_full_size():
    """|dQ| and |dK| reach ~23 here, where bf16's half-ulp (0.0625) alone is
    past 5e-2, so dQ, dK, dV are checked at 5e-2 as float32 outputs (same
    accumulation).  With bf16 storage dV (|dV| < 16, half-ulp 0.031) is still
    held to 5e-2; the bf16 dQ and dK are reported against the bf16-rounded
    oracle value."""
    w = WORKLOADS[3]
    import torch
    inp, scale, out = _run(w, {"": torch.float32, "_bf16": None})
    _check_properties(w, out)
    _check_properties(w, out, "_bf16")
    outputs = {n: _host(out[n]) for n in ("o", "lse", "dq", "dk", "dv")}
    outputs.update({n: _host(out[n]) for n in ("dq_bf16", "dk_bf16", "dv_bf16")})
    worst, fails = check_heads(inp, outputs, _all_heads(inp), scale, w.causal, TOL["bf16"],
                               report=("dq_bf16", "dk_bf16", "dv_bf16"))
    _assert_clean(worst, fails, "BERT shape, all 1024 heads")
    assert worst["dv_bf16_vs_f64"] <= TOL["bf16"]["grad"], worst["dv_bf16_vs_f64"]


LONG_HEADS = [(0, 0), (0, 5), (0, 10), (0, 15), (0, 21), (0, 31), (1, 0), (1, 13), (1, 26),
              (2, 7), (2, 19), (2, 31), (3, 0), (3, 12), (3, 24), (3, 31)]


def test_long_context_full_size():
    w = WORKLOADS[4]
    inp, scale, out = _run(w, {"": None})
    _check_properties(w, out)
    assert (0, 0) in LONG_HEADS and (inp.B - 1, inp.H - 1) in LONG_HEADS
    outputs = {n: _host(out[n]) for n in ("o", "lse", "dq", "dk", "dv")}
    worst, fails = check_heads(inp, outputs, LONG_HEADS, scale, w.causal, TOL["bf16"],
                               workers=workers_for(4 << 30, cap=8))
    _assert_clean(worst, fails, "long context, 16 heads")
