"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory
at call time.  Its D scratch is a fixed array inside the library instead of a
caller workspace; its results must match fa_bwd's.

Kept in a file of its own that pytest collects last, and written so it passes
both alone in a fresh process and after the other GPU tests."""

import pytest

from exact_attention_fwd_gb300.inputs import torch_to_f64
from tests.gpu_util import TOL, make, require_gpu

pytestmark = pytest.mark.gpu


def _grads_both_ways(inp, causal, grad_f32=False):
    torch = require_gpu()
    from exact_attention_fwd_gb300 import _lib, api
    dev = torch.device("cuda", 0)
    q, k, v, do = (inp.torch(t, dev) for t in ("q", "k", "v", "do"))
    o, lse = api.forward(q, k, v, causal=causal)
    gdt = torch.float32 if grad_f32 else q.dtype
    ref = api.backward(q, k, v, o, lse, do, causal=causal, grad_dtype=gdt)
    assert api.sync_status() == 0
    got = [torch.full_like(t, float("nan")) for t in ref]
    dtype = _lib.FA_DTYPE_BF16 if q.dtype == torch.bfloat16 else _lib.FA_DTYPE_F32
    gcode = _lib.FA_DTYPE_F32 if gdt == torch.float32 else dtype
    B, N, H, d = q.shape
    st = _lib.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                             lse.data_ptr(), do.data_ptr(), got[0].data_ptr(), got[1].data_ptr(),
                             got[2].data_ptr(), B, H, N, d, 1.0 / d ** 0.5, int(causal), dtype,
                             gcode, torch.cuda.current_stream().cuda_stream)
    assert st == _lib.FA_OK, _lib.status_string(st)
    assert api.sync_status() == 0
    return ref, got


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_matches_fa_bwd_on_two_calls_in_a_row(dtype):
    """Two calls in a row, on different inputs and shapes, each against fa_bwd
    with a caller workspace; the second call also shows that the scratch left
    over from the first does not leak into its results."""
    tol = TOL[dtype]["grad"]
    for call, (B, H, N, d, causal, seed) in enumerate(
            [(2, 3, 300, 64, True, 11000), (1, 2, 517, 128 if dtype == "bf16" else 64, False,
                                            11001)]):
        inp = make(B, H, N, d, dtype, seed)
        ref, got = _grads_both_ways(inp, causal)
        for name, r, g in zip(("dq", "dk", "dv"), ref, got):
            err = float((torch_to_f64(g) - torch_to_f64(r)).__abs__().max())
            assert err <= tol, f"call {call + 1}: {name} differs from fa_bwd by {err:.3e}"


def test_noalloc_fp32_gradients():
    inp = make(1, 2, 333, 64, "bf16", 11002, sigma={"q": 4.0, "k": 4.0})
    ref, got = _grads_both_ways(inp, causal=True, grad_f32=True)
    for r, g in zip(ref, got):
        assert float((g - r).abs().max()) <= TOL["bf16"]["grad"]


def test_noalloc_rejects_sizes_beyond_its_scratch():
    require_gpu()
    from exact_attention_fwd_gb300 import _lib
    fake = 1 << 20
    B, H, N = 1, 64, (_lib.FA_BWD_NOALLOC_MAX_ROWS // 64) + 1   # one row over the limit
    st = _lib.fa_bwd_noalloc(fake, 2 * fake, 3 * fake, 4 * fake, 5 * fake, 6 * fake, 8 * fake,
                             10 * fake, 12 * fake, B, H, N, 64, 0.125, 1, _lib.FA_DTYPE_BF16,
                             _lib.FA_DTYPE_BF16, None)
    assert st == _lib.FA_ERR_UNSUPPORTED


def test_noalloc_allocates_no_device_memory():
    """The property the entry point exists for: around warm calls (the first
    call on a device looks up the scratch array's address), neither the
    driver's free device memory nor torch's allocated bytes change.  The two
    calls use 1800 and then 400 rows, so the second finds the first's larger
    scratch contents and must not read them."""
    torch = require_gpu()
    from exact_attention_fwd_gb300 import _lib, api
    dev = torch.device("cuda", 0)
    cases = []
    for B, H, N, causal, seed in [(2, 3, 300, True, 11010), (1, 2, 200, False, 11011)]:
        inp = make(B, H, N, 64, "bf16", seed)
        q, k, v, do = (inp.torch(t, dev) for t in ("q", "k", "v", "do"))
        o, lse = api.forward(q, k, v, causal=causal)
        ref = api.backward(q, k, v, o, lse, do, causal=causal)
        outs = [torch.full_like(q, float("nan")) for _ in range(3)]
        cases.append((q, k, v, o, lse, do, outs, ref, causal))
    stream = torch.cuda.current_stream(dev).cuda_stream

    def call(c):
        q, k, v, o, lse, do, outs, _, causal = c
        B, N, H, d = q.shape
        st = _lib.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), do.data_ptr(), outs[0].data_ptr(),
                                 outs[1].data_ptr(), outs[2].data_ptr(), B, H, N, d,
                                 1.0 / d ** 0.5, int(causal), _lib.FA_DTYPE_BF16,
                                 _lib.FA_DTYPE_BF16, stream)
        assert st == _lib.FA_OK, _lib.status_string(st)

    call(cases[0])                        # warm
    torch.cuda.synchronize(dev)
    assert api.sync_status() == 0
    free0, alloc0 = torch.cuda.mem_get_info(dev)[0], torch.cuda.memory_allocated(dev)
    call(cases[0])
    call(cases[1])
    torch.cuda.synchronize(dev)
    assert torch.cuda.mem_get_info(dev)[0] == free0
    assert torch.cuda.memory_allocated(dev) == alloc0
    assert api.sync_status() == 0
    for c in cases:
        for g, r in zip(c[6], c[7]):
            assert float((g.float() - r.float()).abs().max()) <= TOL["bf16"]["grad"]
