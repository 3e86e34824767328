"""Split-KV forward on the GPU (fa_fwd_partial, fa_merge, fa_fwd_splitkv)
against the float64 oracle: the per-slice results against
oracle/split_kv.py element by element, the merged output against the plain
definition (oracle/attention.py), and the merge alone against the oracle's
merge of the same float32 slice results."""

import numpy as np
import pytest

from exact_attention_fwd_gb300.inputs import torch_to_f64
from tests.gpu_util import TOL, compare_fwd, default_scale, make, require_gpu

pytestmark = pytest.mark.gpu

DT = {"bf16": "bfloat16", "f16": "float16"}


def _qkv(inp):
    import torch
    dev = torch.device("cuda", 0)
    return tuple(inp.torch(t, dev) for t in ("q", "k", "v"))


def _read_mask(S, N, kps, causal):
    """[S, N] booleans: row i reads slice s."""
    s = np.arange(S)[:, None]
    i = np.arange(N)[None, :]
    return (s * kps <= i) if causal else np.ones((S, N), dtype=bool)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,d,kps,dtype", [
    (1, 2, 1000, 64, 256, "bf16"),
    (2, 1, 700, 128, 512, "bf16"),
    (1, 3, 300, 8, 256, "f16"),
    (1, 2, 257, 64, 256, "f16"),
    (1, 1, 1, 64, 256, "bf16"),
    (1, 2, 2048, 96, 768, "bf16"),
])
def test_partial_matches_oracle(B, H, N, d, kps, dtype, causal):
    torch = require_gpu()
    from exact_attention_fwd_gb300 import api
    from oracle import checker
    from oracle import split_kv as SK
    inp = make(B, H, N, d, dtype, 13000 + N + d)
    q, k, v = _qkv(inp)
    S = -(-N // kps)
    o_part = torch.full((S, B, N, H, d), float("nan"), device=q.device)
    lse_part = torch.full((S, B, H, N), float("nan"), device=q.device)
    api.forward_partial(q, k, v, kps, scale=default_scale(d), causal=causal, o_part=o_part,
                        lse_part=lse_part)
    assert api.sync_status() == 0
    op = o_part.cpu().double().numpy()
    lp = lse_part.cpu().double().numpy()
    ref_o, ref_l = SK.partials(inp.f64("q"), inp.f64("k"), inp.f64("v"), default_scale(d), causal,
                               kps)
    read = _read_mask(S, N, kps, causal)
    tol = TOL[dtype]
    for s in range(S):
        for b in range(B):
            for h in range(H):
                r = read[s]
                ok_o, e_o, n_o = checker.check(op[s, b, r, h, :], ref_o[s, b, r, h, :], tol["o"])
                ok_l, e_l, n_l = checker.check(lp[s, b, h, r], ref_l[s, b, h, r], tol["lse"])
                assert ok_o, f"O slice {s} head {(b, h)}: {e_o:.3e}, {n_o} mismatches"
                assert ok_l, f"L slice {s} head {(b, h)}: {e_l:.3e}, {n_l} mismatches"
                # entries of slices a row does not read are left untouched
                assert np.isnan(op[s, b, ~r, h, :]).all()
                assert np.isnan(lp[s, b, h, ~r]).all()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("num_splits", [1, 2, 3, 8])
def test_splitkv_matches_oracle_forward(num_splits, causal):
    require_gpu()
    from exact_attention_fwd_gb300 import api
    inp = make(2, 2, 1100, 64, "bf16", 13500 + num_splits)
    q, k, v = _qkv(inp)
    o, lse = api.forward_splitkv(q, k, v, num_splits, scale=default_scale(64), causal=causal)
    assert api.sync_status() == 0
    compare_fwd(inp, o, lse, causal, default_scale(64))


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_splitkv_long_few_heads(dtype):
    """Few heads, long N (the case the slices are for): every row of 2 heads."""
    require_gpu()
    from exact_attention_fwd_gb300 import api
    inp = make(1, 2, 8192, 128, dtype, 13600)
    q, k, v = _qkv(inp)
    o, lse = api.forward_splitkv(q, k, v, 8, scale=default_scale(128), causal=True)
    assert api.sync_status() == 0
    compare_fwd(inp, o, lse, True, default_scale(128))


@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_merge_matches_oracle_merge(causal, out):
    """fa_merge on slice results made by the oracle (rounded to float32), with
    a slice of -inf rows and NaN in every entry no row reads."""
    torch = require_gpu()
    from exact_attention_fwd_gb300 import api
    from oracle import checker
    from oracle import split_kv as SK
    B, H, N, d, kps = 2, 3, 900, 64, 256
    rng = np.random.default_rng(13700)
    q, k, v = (rng.normal(0, 1.5, (B, N, H, d)) for _ in range(3))
    op, lp = SK.partials(q, k, v, 0.2, causal, kps)
    S = op.shape[0]
    # slice 1 of head (1, 2): -inf rows (contribute nothing), NaN O (never read)
    lp[1, 1, 2, :] = np.where(np.isnan(lp[1, 1, 2, :]), np.nan, -np.inf)
    op[1, 1, :, 2, :] = np.nan
    op32, lp32 = op.astype(np.float32), lp.astype(np.float32)
    dev = torch.device("cuda", 0)
    o_t = torch.from_numpy(op32).to(dev)
    l_t = torch.from_numpy(lp32).to(dev)
    dt = torch.float32 if out == "f32" else torch.bfloat16
    o, lse = api.merge(o_t, l_t, kps, causal=causal, dtype=dt)
    assert api.sync_status() == 0
    want_o, want_l = SK.merge(op32.astype(np.float64), lp32.astype(np.float64), kps, causal)
    got_o = torch_to_f64(o)
    got_l = lse.cpu().double().numpy()
    assert np.isfinite(got_o).all()
    tol_o = TOL["f32"]["o"] if out == "f32" else TOL["bf16"]["o"]
    ok, e, n = checker.check(got_o, want_o, tol_o)
    assert ok, f"O: {e:.3e}, {n} mismatches"
    ok, e, n = checker.check(got_l, want_l, 1e-5)
    assert ok, f"L: {e:.3e}, {n} mismatches"
    assert S == 4


def test_merge_rows_without_contribution():
    """A row whose every slice is -inf gets O = 0 and L = -inf."""
    torch = require_gpu()
    from exact_attention_fwd_gb300 import api
    dev = torch.device("cuda", 0)
    S, B, N, H, d = 3, 1, 5, 2, 8
    o_part = torch.full((S, B, N, H, d), float("nan"), device=dev)
    lse_part = torch.full((S, B, H, N), float("-inf"), device=dev)
    lse_part[0, 0, 0, 1] = 0.5
    o_part[0, 0, 1, 0, :] = 2.0
    o, lse = api.merge(o_part, lse_part, 256, causal=False, dtype=torch.float32)
    assert api.sync_status() == 0
    o = o.cpu().numpy()
    lse = lse.cpu().numpy()
    assert (o[0, 1, 0, :] == 2.0).all() and lse[0, 0, 1] == np.float32(0.5)
    mask = np.ones((N, H), dtype=bool)
    mask[1, 0] = False
    assert (o[0][mask] == 0.0).all()
    assert np.isneginf(lse[0].T[mask]).all()


def test_partial_bounded_wait_self_test():
    """The split-KV pass runs the forward kernel in split mode: the self-test
    switch makes its first wait time out and report FA_ERR_TIMEOUT."""
    import os
    torch = require_gpu()
    from exact_attention_fwd_gb300 import _lib, api
    inp = make(1, 2, 600, 64, "bf16", 13800)
    q, k, v = _qkv(inp)
    os.environ["FA_SELFTEST_WAIT_TIMEOUT"] = "1"
    try:
        api.forward_partial(q, k, v, 256, causal=True)
        st = api.sync_status()
    finally:
        del os.environ["FA_SELFTEST_WAIT_TIMEOUT"]
    assert st == _lib.FA_ERR_TIMEOUT
    assert api.sync_status() == 0
    o, lse = api.forward_splitkv(q, k, v, 2, causal=True)
    assert api.sync_status() == 0
    compare_fwd(inp, o, lse, True, default_scale(64))
