"""The unfused comparison forward (fa_fwd_unfused: S to global memory, a row
softmax, P V) against the float64 oracle on the same seeded inputs."""

import pytest

from tests.gpu_util import compare_fwd, default_scale, make, require_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,d,dtype", [
    (2, 2, 300, 64, "bf16"),
    (1, 3, 129, 128, "bf16"),
    (1, 2, 1, 64, "bf16"),
    (2, 1, 257, 40, "f16"),
    (1, 2, 1024, 64, "f16"),
])
def test_unfused_matches_oracle(B, H, N, d, dtype, causal):
    torch = require_gpu()
    from exact_attention_fwd_gb300 import api
    inp = make(B, H, N, d, dtype, 15000 + N + d)
    dev = torch.device("cuda", 0)
    q, k, v = (inp.torch(t, dev) for t in ("q", "k", "v"))
    o, lse = api.forward_unfused(q, k, v, scale=default_scale(d), causal=causal)
    assert api.sync_status() == 0
    compare_fwd(inp, o, lse, causal, default_scale(d))


def test_unfused_large_scores():
    """Q, K ~ N(0, 4^2): wide score range, as in the BERT-shaped workload."""
    torch = require_gpu()
    from exact_attention_fwd_gb300 import api
    inp = make(1, 4, 512, 64, "bf16", 15500, sigma={"q": 4.0, "k": 4.0})
    dev = torch.device("cuda", 0)
    q, k, v = (inp.torch(t, dev) for t in ("q", "k", "v"))
    for causal in (False, True):
        o, lse = api.forward_unfused(q, k, v, causal=causal)
        assert api.sync_status() == 0
        compare_fwd(inp, o, lse, causal, default_scale(64))
