"""Named single-GPU workloads for timing and profiling the entry points.

``python -m exact_attention_fwd_gb300.cases <name> [--reps R]`` builds seeded
N(0, 1) inputs on ``cuda:0``, makes one untimed call, then times ``R`` calls
with CUDA events and prints one line: the case, its shape and the mean time
per call.  The captures in ``profiles/`` name these cases, so every profile
can be re-run from the committed tree.  The first call is the warm-up, so an
``ncu -s 1 -c 1`` capture of a one-kernel case takes a warm launch.

Cases (FLOP counted as 4 B H d times the visible (query, key) pairs for a
forward):

* ``long_fwd``: B1 H32 N8192 d128 causal bf16, ``forward``;
* ``gpt2_unfused``: B8 H16 N1024 d64 causal bf16, ``forward`` then
  ``forward_unfused`` per repetition;
* ``tf32x3``: B8 H16 N1024 d64 causal float32, ``forward_tf32x3`` (split pass
  plus one tensor-core kernel);
* ``tf32x3_bwd``: B8 H16 N1024 d64 causal float32, ``backward_tf32x3`` (split
  passes, the D pre-pass, the dQ kernel and the dK/dV kernel; FLOP 2.5 times
  the forward's);
* ``splitkv``: B1 H1 N32768 d128 causal bf16, ``forward_splitkv`` with 8 key
  slices (partial forward plus merge);
* ``bert_fwd`` / ``bert_bwd``: B64 H16 N512 d64 non-causal bf16, Q and K with
  standard deviation 4, ``forward`` / ``backward`` (backward FLOP 2.5 times the
  forward's);
* ``long4_fwd`` / ``long4_bwd``: B4 H32 N8192 d128 causal bf16, ``forward`` /
  ``backward``.
"""
import argparse

import torch

from . import api


def _pairs(N, causal):
    return N * (N + 1) // 2 if causal else N * N


def _inputs(shape, dtype, dev, seed=0, count=3):
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    return [torch.randn(*shape, device=dev, generator=g).to(dtype) for _ in range(count)]


def _case_long_fwd(dev):
    B, H, N, d = 1, 32, 8192, 128
    q, k, v = _inputs((B, N, H, d), torch.bfloat16, dev)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, device=dev)
    return (B, H, N, d), 4.0 * B * H * d * _pairs(N, True), \
        lambda: api.forward(q, k, v, causal=True, out=o, lse=lse)


def _case_gpt2_unfused(dev):
    B, H, N, d = 8, 16, 1024, 64
    q, k, v = _inputs((B, N, H, d), torch.bfloat16, dev)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, device=dev)
    o2 = torch.empty_like(q)
    lse2 = torch.empty(B, H, N, device=dev)
    ws = api.unfused_workspace(B, H, N, d, dev)

    def run():
        api.forward(q, k, v, causal=True, out=o, lse=lse)
        api.forward_unfused(q, k, v, causal=True, out=o2, lse=lse2, ws=ws)
    return (B, H, N, d), 2 * 4.0 * B * H * d * _pairs(N, True), run


def _case_tf32x3(dev):
    B, H, N, d = 8, 16, 1024, 64
    q, k, v = _inputs((B, N, H, d), torch.float32, dev)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, device=dev)
    ws = torch.empty(api._lib.fa_fwd_tf32x3_workspace_size(B, H, N, d), dtype=torch.uint8,
                     device=dev)
    return (B, H, N, d), 4.0 * B * H * d * _pairs(N, True), \
        lambda: api.forward_tf32x3(q, k, v, causal=True, out=o, lse=lse, ws=ws)


def _case_tf32x3_bwd(dev):
    B, H, N, d = 8, 16, 1024, 64
    q, k, v, do = _inputs((B, N, H, d), torch.float32, dev, count=4)
    o, lse = api.forward(q, k, v, causal=True)
    ws = torch.empty(api._lib.fa_bwd_tf32x3_workspace_size(B, H, N, d), dtype=torch.uint8,
                     device=dev)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    return (B, H, N, d), 2.5 * 4.0 * B * H * d * _pairs(N, True), \
        lambda: api.backward_tf32x3(q, k, v, o, lse, do, causal=True, ws=ws, dq=dq, dk=dk, dv=dv)


def _case_splitkv(dev):
    B, H, N, d, S = 1, 1, 32768, 128, 8
    q, k, v = _inputs((B, N, H, d), torch.bfloat16, dev)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, device=dev)
    ws = api.splitkv_workspace(B, H, N, d, S, dev)
    return (B, H, N, d), 4.0 * B * H * d * _pairs(N, True), \
        lambda: api.forward_splitkv(q, k, v, S, causal=True, out=o, lse=lse, ws=ws)


def _fwd_bwd_pair(B, H, N, d, causal, qk_std, dev, backward):
    q, k, v, do = _inputs((B, N, H, d), torch.float32, dev, count=4)
    q, k = (t * qk_std for t in (q, k))
    q, k, v, do = (t.to(torch.bfloat16) for t in (q, k, v, do))
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, device=dev)
    flop = 4.0 * B * H * d * _pairs(N, causal)
    if not backward:
        return (B, H, N, d), flop, lambda: api.forward(q, k, v, causal=causal, out=o, lse=lse)
    api.forward(q, k, v, causal=causal, out=o, lse=lse)
    ws = api.workspace(B, H, N, dev)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    return (B, H, N, d), 2.5 * flop, lambda: api.backward(
        q, k, v, o, lse, do, causal=causal, ws=ws, dq=dq, dk=dk, dv=dv)


CASES = {
    "long_fwd": _case_long_fwd,
    "gpt2_unfused": _case_gpt2_unfused,
    "tf32x3": _case_tf32x3,
    "tf32x3_bwd": _case_tf32x3_bwd,
    "splitkv": _case_splitkv,
    "bert_fwd": lambda dev: _fwd_bwd_pair(64, 16, 512, 64, False, 4.0, dev, False),
    "bert_bwd": lambda dev: _fwd_bwd_pair(64, 16, 512, 64, False, 4.0, dev, True),
    "long4_fwd": lambda dev: _fwd_bwd_pair(4, 32, 8192, 128, True, 1.0, dev, False),
    "long4_bwd": lambda dev: _fwd_bwd_pair(4, 32, 8192, 128, True, 1.0, dev, True),
}


def run_case(name, reps=5):
    """Run case ``name`` once untimed and ``reps`` times timed; returns
    (shape, mean milliseconds per call, TFLOP/s)."""
    dev = torch.device("cuda", 0)
    shape, flop, fn = CASES[name](dev)
    fn()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(reps):
        fn()
    end.record()
    end.synchronize()
    status = api.sync_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after case {name}")
    ms = start.elapsed_time(end) / reps
    return shape, ms, flop / (ms * 1e-3) / 1e12


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("case", choices=sorted(CASES))
    ap.add_argument("--reps", type=int, default=5)
    a = ap.parse_args()
    (B, H, N, d), ms, tf = run_case(a.case, a.reps)
    print(f"{a.case} B{B} H{H} N{N} d{d}: {ms * 1e3:.1f} us per call, {tf:.1f} TFLOP/s")


if __name__ == "__main__":
    main()
