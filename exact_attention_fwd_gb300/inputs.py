"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module holds no attention arithmetic.  It draws the inputs, rounds them
to the storage type and hands out two views of the same values:

* the storage form the CUDA path reads (float32, bf16 as uint16 bit
  patterns, or float16), and
* the exact float64 values of that storage form, for the CPU oracle.

Recipe: numpy.random.default_rng(seed) draws float64 normals N(0, sigma^2) in
the order Q, K, V, dO, each of shape [B, N, H, d] (the pages' [B, T, C] with
C = H * d); each is cast to float32, then for bf16 rounded to nearest-even to
bf16, for f16 rounded to nearest-even to float16 (numpy's conversion).  Seeds
are 1000 * workload index + sub-shape index.
"""

import numpy as np

TENSORS = ("q", "k", "v", "do")


def f32_to_bf16_bits(x):
    """Round float32 values to bf16 (round to nearest, ties to even); returns
    the uint16 bit patterns.  Inputs here are finite."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(bits):
    """Exact float64 values of bf16 bit patterns."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


class Inputs:
    """Q, K, V, dO of one workload in storage form and as exact float64."""

    def __init__(self, B, H, N, d, dtype, seed, sigma=None):
        if dtype not in ("f32", "bf16", "f16"):
            raise ValueError(dtype)
        sigma = dict(sigma or {})
        self.B, self.H, self.N, self.d = B, H, N, d
        self.dtype = dtype
        self.seed = seed
        self.sigma = {t: float(sigma.get(t, 1.0)) for t in TENSORS}
        rng = np.random.default_rng(seed)
        self.storage = {}
        for t in TENSORS:
            x = rng.normal(0.0, self.sigma[t], size=(B, N, H, d)).astype(np.float32)
            if dtype == "f32":
                self.storage[t] = x
            elif dtype == "f16":
                self.storage[t] = x.astype(np.float16)
            else:
                self.storage[t] = f32_to_bf16_bits(x)

    def f64(self, name):
        """Exact float64 values of tensor `name` ([B, N, H, d])."""
        x = self.storage[name]
        return bf16_bits_to_f64(x) if self.dtype == "bf16" else x.astype(np.float64)

    def head_f64(self, name, b, h):
        """Exact float64 values of one head of tensor `name` ([N, d])."""
        x = self.storage[name][b, :, h, :]
        return bf16_bits_to_f64(x) if self.dtype == "bf16" else x.astype(np.float64)

    def torch(self, name, device):
        """The storage form as a torch tensor on `device` (float32, bfloat16 or
        float16)."""
        import torch
        x = self.storage[name]
        if self.dtype in ("f32", "f16"):
            return torch.from_numpy(np.ascontiguousarray(x)).to(device)
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16))
        return t.view(torch.bfloat16).to(device)


def torch_to_f64(t):
    """Exact float64 numpy copy of a float32 / bfloat16 / float16 torch tensor."""
    import torch
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return bf16_bits_to_f64(t.view(torch.int16).numpy().view(np.uint16))
    return t.to(torch.float64).numpy()
