"""torch-tensor front end of the C ABI (argument marshalling only).

torch supplies device memory and the current stream; the library's kernels do
all the work.  Errors from the library raise _lib.FaError.
"""

import math

import torch

from . import _lib

_DTYPES = {torch.float32: _lib.FA_DTYPE_F32, torch.bfloat16: _lib.FA_DTYPE_BF16,
           torch.float16: _lib.FA_DTYPE_F16}


def _check(t, name, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _stream_handle(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def forward(q, k, v, scale=None, causal=False, out=None, lse=None, stream=None):
    """O, LSE = attention(q, k, v).  q, k, v: [B, N, H, d] float32, bfloat16 or float16."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check(t, name, q.dtype)
    if q.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {q.dtype}")
    if q.shape != k.shape or q.shape != v.shape or q.dim() != 4:
        raise ValueError("q, k, v must share one [B, N, H, d] shape")
    B, N, H, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check(out, "out", q.dtype)
    _check(lse, "lse", torch.float32)
    st = _lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                     B, H, N, d, scale, causal, _DTYPES[q.dtype], _stream_handle(stream))
    if st != _lib.FA_OK:
        raise _lib.FaError(st, "fa_fwd")
    return out, lse


def workspace(B, H, N, device):
    """A device workspace tensor sized for fa_bwd."""
    n = _lib.fa_bwd_workspace_size(B, H, N)
    return torch.empty(n, dtype=torch.uint8, device=device)


def backward(q, k, v, o, lse, do, scale=None, causal=False, grad_dtype=None, ws=None,
             dq=None, dk=None, dv=None, stream=None, phase=None):
    """dQ, dK, dV of attention given the forward's O and LSE and the incoming dO."""
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do)):
        _check(t, name, q.dtype)
    _check(lse, "lse", torch.float32)
    B, N, H, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    gdt = q.dtype if grad_dtype is None else grad_dtype
    if ws is None:
        ws = workspace(B, H, N, q.device)
    dq = torch.empty(q.shape, dtype=gdt, device=q.device) if dq is None else dq
    dk = torch.empty(q.shape, dtype=gdt, device=q.device) if dk is None else dk
    dv = torch.empty(q.shape, dtype=gdt, device=q.device) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check(t, name, gdt)
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
            do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, scale,
            causal, _DTYPES[q.dtype], _DTYPES[gdt], ws.data_ptr(), ws.numel(),
            _stream_handle(stream))
    if phase is None:
        st = _lib.fa_bwd(*args)
    else:
        st = _lib.fa_bwd_phase(phase, *args)
    if st != _lib.FA_OK:
        raise _lib.FaError(st, "fa_bwd" if phase is None else f"fa_bwd_phase({phase})")
    return dq, dk, dv


def _check_qkv(q, k, v):
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check(t, name, q.dtype)
    if q.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {q.dtype}")
    if q.shape != k.shape or q.shape != v.shape or q.dim() != 4:
        raise ValueError("q, k, v must share one [B, N, H, d] shape")


def forward_partial(q, k, v, keys_per_split, scale=None, causal=False, o_part=None,
                    lse_part=None, stream=None):
    """Attention of every row over each key slice alone (fa_fwd_partial).

    Returns (o_part [S, B, N, H, d] float32, lse_part [S, B, H, N] float32),
    S = ceil(N / keys_per_split); entries of slices a row does not read (causal:
    slices that start after the row) are left as they were.
    """
    _check_qkv(q, k, v)
    B, N, H, d = q.shape
    S = -(-N // keys_per_split)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if o_part is None:
        o_part = torch.empty((S, B, N, H, d), dtype=torch.float32, device=q.device)
    if lse_part is None:
        lse_part = torch.empty((S, B, H, N), dtype=torch.float32, device=q.device)
    _check(o_part, "o_part", torch.float32)
    _check(lse_part, "lse_part", torch.float32)
    st = _lib.fa_fwd_partial(q.data_ptr(), k.data_ptr(), v.data_ptr(), o_part.data_ptr(),
                             lse_part.data_ptr(), B, H, N, d, scale, causal, _DTYPES[q.dtype],
                             keys_per_split, _stream_handle(stream))
    if st != _lib.FA_OK:
        raise _lib.FaError(st, "fa_fwd_partial")
    return o_part, lse_part


def merge(o_part, lse_part, keys_per_split, causal=False, dtype=torch.bfloat16, out=None,
          lse=None, stream=None):
    """Merge per-slice results into (O [B, N, H, d] of `dtype`, LSE [B, H, N]) (fa_merge)."""
    _check(o_part, "o_part", torch.float32)
    _check(lse_part, "lse_part", torch.float32)
    if o_part.dim() != 5:
        raise ValueError("o_part must be [S, B, N, H, d]")
    S, B, N, H, d = o_part.shape
    if tuple(lse_part.shape) != (S, B, H, N):
        raise ValueError("lse_part must be [S, B, H, N]")
    if dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {dtype}")
    if out is None:
        out = torch.empty((B, N, H, d), dtype=dtype, device=o_part.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=o_part.device)
    _check(out, "out", dtype)
    _check(lse, "lse", torch.float32)
    st = _lib.fa_merge(o_part.data_ptr(), lse_part.data_ptr(), S, keys_per_split, causal,
                       out.data_ptr(), lse.data_ptr(), B, H, N, d, _DTYPES[dtype],
                       _stream_handle(stream))
    if st != _lib.FA_OK:
        raise _lib.FaError(st, "fa_merge")
    return out, lse


def splitkv_workspace(B, H, N, d, num_splits, device):
    """A device workspace tensor sized for fa_fwd_splitkv."""
    n = _lib.fa_fwd_splitkv_workspace_size(B, H, N, d, num_splits)
    return torch.empty(n, dtype=torch.uint8, device=device)


def forward_splitkv(q, k, v, num_splits, scale=None, causal=False, out=None, lse=None, ws=None,
                    stream=None):
    """O, LSE = attention(q, k, v) as key slices then a merge (fa_fwd_splitkv)."""
    _check_qkv(q, k, v)
    B, N, H, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = splitkv_workspace(B, H, N, d, num_splits, q.device)
    _check(out, "out", q.dtype)
    _check(lse, "lse", torch.float32)
    st = _lib.fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                             lse.data_ptr(), B, H, N, d, scale, causal, _DTYPES[q.dtype],
                             num_splits, ws.data_ptr(), ws.numel(), _stream_handle(stream))
    if st != _lib.FA_OK:
        raise _lib.FaError(st, "fa_fwd_splitkv")
    return out, lse


def _check_host(t, name, dtype):
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def host_workspace(batch_chunk, H, N, d, dtype, grad_dtype, device):
    """A device workspace tensor sized for fwd_bwd_host."""
    n = _lib.fa_fwd_bwd_host_workspace_size(batch_chunk, H, N, d, _DTYPES[dtype], _DTYPES[grad_dtype])
    return torch.empty(n, dtype=torch.uint8, device=device)


def fwd_bwd_host(q, k, v, do, batch_chunk, scale=None, causal=False, grad_dtype=None, out=None,
                 ws=None, device=None, stream=None):
    """Forward and backward on host tensors (fa_fwd_bwd_host): copies in, both
    passes and copies out, pipelined over chunks of `batch_chunk` sequences.

    q, k, v, do: [B, N, H, d] CPU tensors (pinned for overlap).  Returns the
    host tensors (o, lse, dq, dk, dv), complete once `stream` is synchronised.
    """
    for name, t in (("q", q), ("k", k), ("v", v), ("do", do)):
        _check_host(t, name, q.dtype)
    if q.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {q.dtype}")
    B, N, H, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    gdt = q.dtype if grad_dtype is None else grad_dtype
    device = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    bc = min(batch_chunk, B)
    if ws is None:
        ws = host_workspace(bc, H, N, d, q.dtype, gdt, device)
    if out is None:
        pin = q.is_pinned()
        out = (torch.empty(q.shape, dtype=q.dtype, pin_memory=pin),
               torch.empty((B, H, N), dtype=torch.float32, pin_memory=pin),
               *(torch.empty(q.shape, dtype=gdt, pin_memory=pin) for _ in range(3)))
    o, lse, dq, dk, dv = out
    _check_host(o, "o", q.dtype)
    _check_host(lse, "lse", torch.float32)
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check_host(t, name, gdt)
    st = _lib.fa_fwd_bwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(),
                              o.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                              dv.data_ptr(), B, H, N, d, scale, causal, _DTYPES[q.dtype],
                              _DTYPES[gdt], batch_chunk, ws.data_ptr(), ws.numel(),
                              _stream_handle(stream))
    if st != _lib.FA_OK:
        raise _lib.FaError(st, "fa_fwd_bwd_host")
    return o, lse, dq, dk, dv


def unfused_workspace(B, H, N, d, device):
    """A device workspace tensor sized for forward_unfused (holds S, B H N^2 floats)."""
    n = _lib.fa_fwd_unfused_workspace_size(B, H, N, d)
    return torch.empty(n, dtype=torch.uint8, device=device)


def forward_unfused(q, k, v, scale=None, causal=False, out=None, lse=None, ws=None, stream=None):
    """The unfused forward (fa_fwd_unfused): S to global memory, a row softmax,
    then P V; a comparison for forward()."""
    _check_qkv(q, k, v)
    B, N, H, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = unfused_workspace(B, H, N, d, q.device)
    _check(out, "out", q.dtype)
    _check(lse, "lse", torch.float32)
    st = _lib.fa_fwd_unfused(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                             lse.data_ptr(), B, H, N, d, scale, causal, _DTYPES[q.dtype],
                             ws.data_ptr(), ws.numel(), _stream_handle(stream))
    if st != _lib.FA_OK:
        raise _lib.FaError(st, "fa_fwd_unfused")
    return out, lse


def forward_tf32x3(q, k, v, scale=None, causal=False, out=None, lse=None, ws=None, stream=None):
    """float32 O, LSE = attention(q, k, v) on the tensor cores (fa_fwd_tf32x3, d <= 128)."""
    _check_qkv(q, k, v)
    if q.dtype != torch.float32:
        raise ValueError("forward_tf32x3 takes float32 tensors")
    B, N, H, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = torch.empty(_lib.fa_fwd_tf32x3_workspace_size(B, H, N, d), dtype=torch.uint8,
                         device=q.device)
    _check(out, "out", torch.float32)
    _check(lse, "lse", torch.float32)
    st = _lib.fa_fwd_tf32x3(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                            lse.data_ptr(), B, H, N, d, scale, causal, ws.data_ptr(), ws.numel(),
                            _stream_handle(stream))
    if st != _lib.FA_OK:
        raise _lib.FaError(st, "fa_fwd_tf32x3")
    return out, lse


def backward_tf32x3(q, k, v, o, lse, do, scale=None, causal=False, ws=None, dq=None, dk=None,
                    dv=None, stream=None):
    """float32 dQ, dK, dV on the tensor cores (fa_bwd_tf32x3, d <= 64)."""
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do)):
        _check(t, name, torch.float32)
    _check(lse, "lse", torch.float32)
    if q.shape != k.shape or q.shape != v.shape or q.shape != o.shape or q.shape != do.shape:
        raise ValueError("q, k, v, o, do must share one [B, N, H, d] shape")
    B, N, H, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if ws is None:
        ws = torch.empty(_lib.fa_bwd_tf32x3_workspace_size(B, H, N, d), dtype=torch.uint8,
                         device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check(t, name, torch.float32)
    st = _lib.fa_bwd_tf32x3(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                            lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                            dv.data_ptr(), B, H, N, d, scale, causal, ws.data_ptr(), ws.numel(),
                            _stream_handle(stream))
    if st != _lib.FA_OK:
        raise _lib.FaError(st, "fa_bwd_tf32x3")
    return dq, dk, dv


def sync_status(stream=None):
    """Synchronise and return (and clear) the device status word."""
    return _lib.fa_sync_status(_stream_handle(stream))
