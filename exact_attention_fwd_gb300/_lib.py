"""ctypes binding of libfa.so: the C ABI of include/fa.h under the same names.

Argument marshalling only.  Every step of the computation runs in the
library's CUDA kernels; nothing here computes attention, and there is no
fallback: if libfa.so is missing the calls raise.
"""

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfa.so")

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(5)
FA_DTYPE_F32, FA_DTYPE_BF16, FA_DTYPE_F16 = range(3)

EXPORTS = ("fa_fwd", "fa_bwd", "fa_bwd_phase", "fa_bwd_workspace_size", "fa_sync_status",
           "fa_status_string", "fa_bwd_noalloc", "fa_fwd_partial", "fa_merge",
           "fa_fwd_splitkv_keys_per_split", "fa_fwd_splitkv_workspace_size", "fa_fwd_splitkv",
           "fa_fwd_bwd_host_workspace_size", "fa_fwd_bwd_host", "fa_fwd_unfused_workspace_size",
           "fa_fwd_unfused", "fa_fwd_tf32x3_workspace_size", "fa_fwd_tf32x3",
           "fa_bwd_tf32x3_workspace_size", "fa_bwd_tf32x3", "fa_bwd_prepass")
FA_BWD_NOALLOC_MAX_ROWS = 1 << 22

_lib = None


class FaError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def load():
    """Load libfa.so (once) and declare the signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is not built; run exact_attention_fwd_gb300.build.build() first")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
    lib.fa_fwd.restype = i
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, i, vp, sz, vp]
    lib.fa_bwd.restype = i
    lib.fa_bwd_phase.argtypes = [i] + lib.fa_bwd.argtypes
    lib.fa_bwd_phase.restype = i
    lib.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, i, vp]
    lib.fa_bwd_noalloc.restype = i
    lib.fa_bwd_workspace_size.argtypes = [i, i, i]
    lib.fa_bwd_workspace_size.restype = sz
    lib.fa_sync_status.argtypes = [vp]
    lib.fa_sync_status.restype = i
    lib.fa_fwd_partial.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, i, vp]
    lib.fa_fwd_partial.restype = i
    lib.fa_merge.argtypes = [vp, vp, i, i, i, vp, vp, i, i, i, i, i, vp]
    lib.fa_merge.restype = i
    lib.fa_fwd_splitkv_keys_per_split.argtypes = [i, i]
    lib.fa_fwd_splitkv_keys_per_split.restype = i
    lib.fa_fwd_splitkv_workspace_size.argtypes = [i, i, i, i, i]
    lib.fa_fwd_splitkv_workspace_size.restype = sz
    lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, i, vp, sz, vp]
    lib.fa_fwd_splitkv.restype = i
    lib.fa_fwd_bwd_host_workspace_size.argtypes = [i, i, i, i, i, i]
    lib.fa_fwd_bwd_host_workspace_size.restype = sz
    lib.fa_fwd_bwd_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, i, i, i,
                                    vp, sz, vp]
    lib.fa_fwd_bwd_host.restype = i
    lib.fa_fwd_unfused_workspace_size.argtypes = [i, i, i, i]
    lib.fa_fwd_unfused_workspace_size.restype = sz
    lib.fa_fwd_unfused.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp, sz, vp]
    lib.fa_fwd_unfused.restype = i
    lib.fa_fwd_tf32x3_workspace_size.argtypes = [i, i, i, i]
    lib.fa_fwd_tf32x3_workspace_size.restype = sz
    lib.fa_fwd_tf32x3.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, sz, vp]
    lib.fa_fwd_tf32x3.restype = i
    lib.fa_bwd_tf32x3_workspace_size.argtypes = [i, i, i, i]
    lib.fa_bwd_tf32x3_workspace_size.restype = sz
    lib.fa_bwd_tf32x3.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, sz, vp]
    lib.fa_bwd_tf32x3.restype = i
    lib.fa_bwd_prepass.argtypes = [i, i]
    lib.fa_bwd_prepass.restype = i
    lib.fa_status_string.argtypes = [i]
    lib.fa_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(s):
    return load().fa_status_string(int(s)).decode()


def fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, stream):
    """Raw call: pointers are ints (device addresses); returns the status."""
    return load().fa_fwd(q, k, v, o, lse, B, H, N, d, float(scale), int(causal), int(dtype),
                         stream)


def fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, dtype, grad_dtype,
           workspace, workspace_bytes, stream):
    return load().fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, float(scale), int(causal),
                         int(dtype), int(grad_dtype), workspace, workspace_bytes, stream)


def fa_bwd_phase(phase, q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, dtype,
                 grad_dtype, workspace, workspace_bytes, stream):
    return load().fa_bwd_phase(int(phase), q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d,
                               float(scale), int(causal), int(dtype), int(grad_dtype), workspace,
                               workspace_bytes, stream)


def fa_bwd_noalloc(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, dtype,
                   grad_dtype, stream):
    """fa_bwd with the library's fixed device scratch instead of a workspace."""
    return load().fa_bwd_noalloc(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, float(scale),
                                 int(causal), int(dtype), int(grad_dtype), stream)


def fa_bwd_prepass(d, dtype):
    """1 if fa_bwd's phase 0 launches the D pre-pass for this d and dtype."""
    return int(load().fa_bwd_prepass(int(d), int(dtype)))


def fa_bwd_workspace_size(B, H, N):
    return int(load().fa_bwd_workspace_size(B, H, N))


def fa_sync_status(stream):
    return load().fa_sync_status(stream)


def fa_fwd_partial(q, k, v, o_part, lse_part, B, H, N, d, scale, causal, dtype, keys_per_split,
                   stream):
    return load().fa_fwd_partial(q, k, v, o_part, lse_part, B, H, N, d, float(scale),
                                 int(causal), int(dtype), int(keys_per_split), stream)


def fa_merge(o_part, lse_part, num_splits, keys_per_split, causal, o, lse, B, H, N, d, dtype,
             stream):
    return load().fa_merge(o_part, lse_part, int(num_splits), int(keys_per_split), int(causal),
                           o, lse, B, H, N, d, int(dtype), stream)


def fa_fwd_splitkv_keys_per_split(N, num_splits):
    return int(load().fa_fwd_splitkv_keys_per_split(N, num_splits))


def fa_fwd_splitkv_workspace_size(B, H, N, d, num_splits):
    return int(load().fa_fwd_splitkv_workspace_size(B, H, N, d, num_splits))


def fa_fwd_splitkv(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, num_splits, workspace,
                   workspace_bytes, stream):
    return load().fa_fwd_splitkv(q, k, v, o, lse, B, H, N, d, float(scale), int(causal),
                                 int(dtype), int(num_splits), workspace, workspace_bytes, stream)


def fa_fwd_bwd_host_workspace_size(batch_chunk, H, N, d, dtype, grad_dtype):
    return int(load().fa_fwd_bwd_host_workspace_size(batch_chunk, H, N, d, int(dtype),
                                                     int(grad_dtype)))


def fa_fwd_bwd_host(q, k, v, dO, o, lse, dq, dk, dv, B, H, N, d, scale, causal, dtype, grad_dtype,
                    batch_chunk, workspace, workspace_bytes, stream):
    """Host pointers for the tensors, a device workspace; see include/fa.h."""
    return load().fa_fwd_bwd_host(q, k, v, dO, o, lse, dq, dk, dv, B, H, N, d, float(scale),
                                  int(causal), int(dtype), int(grad_dtype), int(batch_chunk),
                                  workspace, workspace_bytes, stream)


def fa_fwd_unfused_workspace_size(B, H, N, d):
    return int(load().fa_fwd_unfused_workspace_size(B, H, N, d))


def fa_fwd_unfused(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, workspace, workspace_bytes,
                   stream):
    """The unfused comparison forward (include/fa.h)."""
    return load().fa_fwd_unfused(q, k, v, o, lse, B, H, N, d, float(scale), int(causal),
                                 int(dtype), workspace, workspace_bytes, stream)


def fa_bwd_tf32x3_workspace_size(B, H, N, d):
    return int(load().fa_bwd_tf32x3_workspace_size(B, H, N, d))


def fa_bwd_tf32x3(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, workspace,
                  workspace_bytes, stream):
    """float32 backward on the tensor cores (3xTF32); pointers as integers."""
    return load().fa_bwd_tf32x3(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, float(scale),
                                int(causal), workspace, workspace_bytes, stream)


def fa_fwd_tf32x3_workspace_size(B, H, N, d):
    return int(load().fa_fwd_tf32x3_workspace_size(B, H, N, d))


def fa_fwd_tf32x3(q, k, v, o, lse, B, H, N, d, scale, causal, workspace, workspace_bytes, stream):
    """float32 forward on the tensor cores (include/fa.h)."""
    return load().fa_fwd_tf32x3(q, k, v, o, lse, B, H, N, d, float(scale), int(causal), workspace,
                                workspace_bytes, stream)
