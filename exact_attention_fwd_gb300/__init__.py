"""Fused exact attention (FlashAttention-2 forward and recompute backward) for
GB300 / sm_103a, behind the C ABI of include/fa.h.

    from exact_attention_fwd_gb300 import api
    o, lse = api.forward(q, k, v, causal=True)          # torch CUDA tensors
    dq, dk, dv = api.backward(q, k, v, o, lse, do, causal=True)

Tensors are [B, N, H, d] (float32 or bfloat16), LSE is [B, H, N] float32.
The library (libfa.so) is built in-tree by exact_attention_fwd_gb300.build.
Importing this package does not load it; the first call does, and raises if
it is missing.
"""
