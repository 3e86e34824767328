"""Helpers shared by the GPU parity tests: build/load the library once, run the
CUDA path through the C ABI (via the torch front end), and run the oracle on
the same seeded inputs."""

import math

import numpy as np
import pytest

from exact_attention_fwd_gb300.inputs import Inputs, torch_to_f64

TOL = {  # max-abs tolerances fixed for this operator
    "f32": {"o": 1e-5, "grad": 1e-4, "lse": 1e-4},
    "bf16": {"o": 2e-2, "grad": 5e-2, "lse": 1e-4},
    # fp16 I/O: the 16-bit tolerances (fp32 accumulation in both); fp16's
    # finer significand makes them stricter in effect
    "f16": {"o": 2e-2, "grad": 5e-2, "lse": 1e-4},
}


def require_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_fwd_gb300 import build
    build.build()
    return torch


def run_fwd(inp, causal, scale=None):
    import torch
    from exact_attention_fwd_gb300 import api
    dev = torch.device("cuda", 0)
    q, k, v = (inp.torch(t, dev) for t in ("q", "k", "v"))
    o, lse = api.forward(q, k, v, scale=scale, causal=causal)
    st = api.sync_status()
    assert st == 0, f"device status {st}"
    return o, lse, (q, k, v)


def oracle_fwd_heads(inp, causal, scale, heads):
    from oracle import attention as A
    out = {}
    for b, h in heads:
        out[(b, h)] = A.forward_head(inp.head_f64("q", b, h), inp.head_f64("k", b, h),
                                     inp.head_f64("v", b, h), scale, causal)
    return out


def all_heads(inp):
    return [(b, h) for b in range(inp.B) for h in range(inp.H)]


def compare_fwd(inp, o_gpu, lse_gpu, causal, scale, heads=None, tol=None):
    """Element-by-element comparison on the given heads; returns worst errors."""
    from oracle import checker
    tol = tol or TOL[inp.dtype]
    heads = heads or all_heads(inp)
    ref = oracle_fwd_heads(inp, causal, scale, heads)
    o64 = torch_to_f64(o_gpu)
    l64 = lse_gpu.detach().cpu().double().numpy()
    worst_o = worst_l = 0.0
    for (b, h), (o_ref, l_ref) in ref.items():
        ok_o, e_o, n_o = checker.check(o64[b, :, h, :], o_ref, tol["o"])
        ok_l, e_l, n_l = checker.check(l64[b, h, :], l_ref, tol["lse"])
        assert ok_o, f"O head {(b, h)}: max err {e_o:.3e}, {n_o} mismatches"
        assert ok_l, f"LSE head {(b, h)}: max err {e_l:.3e}, {n_l} mismatches"
        worst_o, worst_l = max(worst_o, e_o), max(worst_l, e_l)
    return worst_o, worst_l


def make(B, H, N, d, dtype, seed, sigma=None):
    return Inputs(B, H, N, d, dtype, seed, sigma)


def default_scale(d):
    return 1.0 / math.sqrt(d)
