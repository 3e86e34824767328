"""The many-heads oracle comparison (tests/fullsize_oracle.py) on the CPU:
the oracle's own results, stored the way the CUDA path stores them, pass on
every head; one planted error in one head gives exactly one failure."""

import numpy as np

from exact_attention_fwd_gb300.inputs import Inputs, f32_to_bf16_bits
from tests.fullsize_oracle import check_heads, workers_for
from tests.gpu_util import TOL


def _oracle_outputs(inp, scale, causal):
    from oracle import attention as A
    q, k, v, do = (inp.f64(t) for t in ("q", "k", "v", "do"))
    o, lse = A.forward(q, k, v, scale, causal)
    dq, dk, dv, _ = A.backward(q, k, v, do, scale, causal)
    bits = lambda x: (f32_to_bf16_bits(x.astype(np.float32)), "bf16")
    return {"o": bits(o), "lse": (lse.astype(np.float32), "f32"), "dq": bits(dq),
            "dk": bits(dk), "dv": (dv.astype(np.float32), "f32")}


def test_pool_passes_oracle_and_catches_one_planted_error():
    inp = Inputs(2, 3, 40, 16, "bf16", seed=77)
    scale = 0.25
    out = _oracle_outputs(inp, scale, True)
    heads = [(b, h) for b in range(2) for h in range(3)]
    worst, fails = check_heads(inp, out, heads, scale, True, TOL["bf16"], workers=2)
    assert not fails, fails
    assert worst["o"] < 2e-2 and worst["lse"] < 1e-4
    dk = out["dk"][0].copy()
    dk[1, 17, 2, 5] ^= np.uint16(0x4000)   # a large change of one bf16 value
    out["dk"] = (dk, "bf16")
    _, fails = check_heads(inp, out, heads, scale, True, TOL["bf16"], workers=2)
    assert len(fails) == 1 and fails[0].startswith("dk head (1, 2)") and "1 mismatches" in fails[0]


def test_workers_for_is_bounded():
    assert 1 <= workers_for(1 << 20) <= 16
    assert workers_for(1 << 60) == 1
