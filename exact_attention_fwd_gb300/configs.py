"""The five synthetic workloads the tests and the benchmark run.

Shapes follow the pages' parity shapes ("Flash Attention 2 — forward pass
notes", section "Parity verification") and the FlashAttention paper's GPT-2
medium / BERT-large attention shapes as quoted on the Lesson K23 facts page
(sources.flashAttention, Figure 2 and section 4).  No model weights or
datasets are involved: the inputs are seeded normals (see inputs.py).
"""

import math
from dataclasses import dataclass, field


@dataclass(frozen=True)
class Shape:
    B: int
    H: int
    N: int
    d: int


@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    shapes: tuple            # tuple of Shape
    dtypes: tuple            # subset of ("f32", "bf16")
    causal: bool
    backward: bool
    sigma: dict = field(default_factory=dict)   # per-tensor std dev (default 1)

    def scale(self, shape):
        return 1.0 / math.sqrt(shape.d)

    def seed(self, sub):
        return 1000 * self.index + sub


WORKLOADS = (
    Workload(0, "single_head_N64_d16_f32", (Shape(1, 1, 64, 16),), ("f32",),
             causal=False, backward=False),
    Workload(1, "causal_sweep",
             (Shape(1, 4, 16, 8), Shape(1, 4, 8, 8), Shape(1, 4, 20, 8),
              Shape(1, 2, 256, 32), Shape(1, 1, 128, 64)),
             ("f32", "bf16"), causal=True, backward=True),
    Workload(2, "gpt2_medium_B64_H16_N1024_d64_causal", (Shape(64, 16, 1024, 64),),
             ("bf16",), causal=True, backward=True),
    Workload(3, "bert_large_B64_H16_N512_d64", (Shape(64, 16, 512, 64),), ("bf16",),
             causal=False, backward=True, sigma={"q": 4.0, "k": 4.0}),
    Workload(4, "long_B4_H32_N8192_d128_causal", (Shape(4, 32, 8192, 128),), ("bf16",),
             causal=True, backward=True),
)

# Extra parity shape: the pages' planned browser check (B=2, T=48, C=24, H=3).
BROWSER_SHAPE = Shape(2, 3, 48, 8)


def flops_fwd(B, H, N, d, causal):
    """4 B H N^2 d, halved when causal."""
    f = 4.0 * B * H * N * N * d
    return f * 0.5 if causal else f


def flops_bwd(B, H, N, d, causal):
    """2.5x the forward count."""
    return 2.5 * flops_fwd(B, H, N, d, causal)


def bytes_fwd(B, H, N, d, elt):
    """Read Q, K, V once, write O and the fp32 LSE."""
    return 4 * B * H * N * d * elt + 4 * B * H * N


def bytes_bwd(B, H, N, d, elt, grad_elt=None):
    """Read Q, K, V, O, dO and LSE; write and read D; write dQ, dK, dV."""
    grad_elt = elt if grad_elt is None else grad_elt
    return 5 * B * H * N * d * elt + 3 * B * H * N * d * grad_elt + 12 * B * H * N


def bytes_dot(B, H, N, d, elt):
    """D pre-pass: read O and dO, write D (fp32)."""
    return 2 * B * H * N * d * elt + 4 * B * H * N
