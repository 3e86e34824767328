"""Host-side checks of the C ABI that need no GPU: the library builds and loads,
exports every function include/fa.h declares, and rejects invalid arguments
before launching anything."""

import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from exact_attention_fwd_gb300 import _lib, build
    build.build()
    return _lib.load()


@pytest.fixture(scope="module")
def fake_lib(lib):
    """The library, for calls with fake device addresses that validation must
    reject before any launch.  Skipped where a CUDA device is visible: if a
    case ever passed validation there, its kernels would touch the fake
    addresses."""
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("fake device addresses are only passed where no GPU is visible")
    except ImportError:
        pass
    return lib


def declared_functions():
    src = open(os.path.join(ROOT, "include", "fa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert {"fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_status_string",
            "fa_sync_status"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    from exact_attention_fwd_gb300 import _lib
    assert _lib.status_string(0) == "FA_OK"
    assert _lib.status_string(4) == "FA_ERR_TIMEOUT"
    assert _lib.status_string(99) == "FA_ERR_UNKNOWN"


def test_bwd_prepass_rule(lib):
    """Phase 0 is empty exactly for 16-bit inputs with d <= 64."""
    from exact_attention_fwd_gb300 import _lib
    for d in (8, 64):
        assert _lib.fa_bwd_prepass(d, _lib.FA_DTYPE_BF16) == 0
        assert _lib.fa_bwd_prepass(d, _lib.FA_DTYPE_F16) == 0
        assert _lib.fa_bwd_prepass(d, _lib.FA_DTYPE_F32) == 1
    for d in (72, 128):
        assert _lib.fa_bwd_prepass(d, _lib.FA_DTYPE_BF16) == 1
        assert _lib.fa_bwd_prepass(d, _lib.FA_DTYPE_F32) == 1


def test_workspace_size(lib):
    from exact_attention_fwd_gb300 import _lib
    assert _lib.fa_bwd_workspace_size(64, 16, 1024) == 64 * 16 * 1024 * 4
    assert _lib.fa_bwd_workspace_size(1, 1, 3) == 256
    assert _lib.fa_bwd_workspace_size(0, 1, 3) == 0


FAKE = 1 << 20   # 16-byte aligned address; validation fails before any use


@pytest.mark.parametrize("kw,want", [
    (dict(q=0), 1),                        # null pointer
    (dict(N=0), 1), (dict(B=-1), 1), (dict(H=0), 1),
    (dict(d=12), 1), (dict(d=0), 1),       # not a multiple of 8
    (dict(d=136), 2),                      # above 128
    (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1),
    (dict(dtype=2, q=FAKE + 8), 1),        # fp16, misaligned
    (dict(dtype=7), 1),
    (dict(q=FAKE + 8), 1),                 # misaligned
    (dict(o=FAKE), 1),                     # output aliases q
])
def test_fwd_rejects_invalid_arguments(fake_lib, kw, want):
    from exact_attention_fwd_gb300 import _lib
    a = dict(q=FAKE, k=2 * FAKE, v=3 * FAKE, o=4 * FAKE, lse=5 * FAKE, B=1, H=1, N=16, d=64,
             scale=0.125, causal=1, dtype=1, stream=None)
    a.update(kw)
    assert _lib.fa_fwd(**a) == want


@pytest.mark.parametrize("kw,want", [
    (dict(workspace=0), 1),
    (dict(workspace_bytes=100), 1),
    (dict(grad_dtype=1, dtype=0), 1),      # bf16 grads of fp32 inputs
    (dict(grad_dtype=2, dtype=1), 1),      # fp16 grads of bf16 inputs
    (dict(dtype=3, grad_dtype=3), 1),      # no such element type
    (dict(dq=FAKE), 1),                    # aliases q
    (dict(dk=8 * FAKE), 1),                # aliases dq
    (dict(workspace=FAKE + 16), 1),        # not 256-byte aligned (and aliases)
])
def test_bwd_rejects_invalid_arguments(fake_lib, kw, want):
    from exact_attention_fwd_gb300 import _lib
    a = dict(q=FAKE, k=2 * FAKE, v=3 * FAKE, o=4 * FAKE, lse=5 * FAKE, dO=6 * FAKE,
             dq=8 * FAKE, dk=10 * FAKE, dv=12 * FAKE, B=1, H=1, N=16, d=64, scale=0.125,
             causal=1, dtype=1, grad_dtype=1, workspace=14 * FAKE, workspace_bytes=4096,
             stream=None)
    a.update(kw)
    assert _lib.fa_bwd(**a) == want


def test_bwd_phase_rejects_bad_phase(fake_lib):
    from exact_attention_fwd_gb300 import _lib
    a = dict(q=FAKE, k=2 * FAKE, v=3 * FAKE, o=4 * FAKE, lse=5 * FAKE, dO=6 * FAKE,
             dq=8 * FAKE, dk=10 * FAKE, dv=12 * FAKE, B=1, H=1, N=16, d=64, scale=0.125,
             causal=1, dtype=1, grad_dtype=1, workspace=14 * FAKE, workspace_bytes=4096,
             stream=None)
    assert _lib.fa_bwd_phase(3, **a) == 1
    assert _lib.fa_bwd_phase(-1, **a) == 1
    a["workspace"] = 0
    assert _lib.fa_bwd_phase(1, **a) == 1


def test_splitkv_sizes(lib):
    from exact_attention_fwd_gb300 import _lib
    assert _lib.fa_fwd_splitkv_keys_per_split(8192, 4) == 2048
    assert _lib.fa_fwd_splitkv_keys_per_split(1000, 3) == 512      # 2 slices used
    assert _lib.fa_fwd_splitkv_keys_per_split(100, 8) == 256
    assert _lib.fa_fwd_splitkv_keys_per_split(0, 2) == 0
    assert _lib.fa_fwd_splitkv_keys_per_split(10, 0) == 0
    # 2 slices of [1, 1000, 2, 64] float32 + 2 slices of [1, 2, 1000] float32
    assert _lib.fa_fwd_splitkv_workspace_size(1, 2, 1000, 64, 3) == 1024000 + 16128
    assert _lib.fa_fwd_splitkv_workspace_size(1, 2, 1000, 64, 0) == 0


@pytest.mark.parametrize("kw,want", [
    (dict(o_part=0), 1),
    (dict(keys_per_split=128), 1),         # not a multiple of 256
    (dict(keys_per_split=0), 1),
    (dict(dtype=0), 2),                    # float32 inputs: not on this path
    (dict(d=136), 2),
    (dict(o_part=FAKE + 8), 1),            # misaligned
    (dict(o_part=FAKE), 1),                # overlaps q
    (dict(lse_part=4 * FAKE + 64), 1),     # overlaps o_part
])
def test_fwd_partial_rejects_invalid_arguments(fake_lib, kw, want):
    from exact_attention_fwd_gb300 import _lib
    a = dict(q=FAKE, k=2 * FAKE, v=3 * FAKE, o_part=4 * FAKE, lse_part=8 * FAKE, B=1, H=1, N=16,
             d=64, scale=0.125, causal=1, dtype=1, keys_per_split=256, stream=None)
    a.update(kw)
    assert _lib.fa_fwd_partial(**a) == want


@pytest.mark.parametrize("kw,want", [
    (dict(lse=0), 1),
    (dict(num_splits=0), 1), (dict(keys_per_split=0), 1),
    (dict(dtype=5), 1),
    (dict(o=FAKE + 4), 1),                 # misaligned
    (dict(o=FAKE + 64), 1),                # overlaps o_part
    (dict(N=0), 1),
])
def test_merge_rejects_invalid_arguments(fake_lib, kw, want):
    from exact_attention_fwd_gb300 import _lib
    a = dict(o_part=FAKE, lse_part=2 * FAKE, num_splits=2, keys_per_split=256, causal=1,
             o=4 * FAKE, lse=5 * FAKE, B=1, H=1, N=16, d=64, dtype=1, stream=None)
    a.update(kw)
    assert _lib.fa_merge(**a) == want


@pytest.mark.parametrize("kw,want", [
    (dict(workspace=0), 1),
    (dict(num_splits=0), 1),
    (dict(workspace_bytes=64), 1),
    (dict(workspace=8 * FAKE + 16), 1),    # not 256-byte aligned
    (dict(workspace=FAKE), 1),             # overlaps q
    (dict(dtype=0), 2),
])
def test_splitkv_rejects_invalid_arguments(fake_lib, kw, want):
    from exact_attention_fwd_gb300 import _lib
    a = dict(q=FAKE, k=2 * FAKE, v=3 * FAKE, o=4 * FAKE, lse=5 * FAKE, B=1, H=1, N=16, d=64,
             scale=0.125, causal=1, dtype=1, num_splits=2, workspace=8 * FAKE,
             workspace_bytes=1 << 20, stream=None)
    a.update(kw)
    assert _lib.fa_fwd_splitkv(**a) == want


def test_host_workspace_size(lib):
    from exact_attention_fwd_gb300 import _lib
    # per slot: 5 bf16 tensors + 3 bf16 gradients of 2x16x2x64, L and D of 2x2x16 floats
    t = 2 * 16 * 2 * 64 * 2
    slot = 8 * t + 256 + 256
    assert _lib.fa_fwd_bwd_host_workspace_size(2, 2, 16, 64, 1, 1) == 2 * slot
    # float32 gradients of bf16 inputs
    slot32 = 5 * t + 3 * 2 * t + 256 + 256
    assert _lib.fa_fwd_bwd_host_workspace_size(2, 2, 16, 64, 1, 0) == 2 * slot32
    assert _lib.fa_fwd_bwd_host_workspace_size(0, 2, 16, 64, 1, 1) == 0
    assert _lib.fa_fwd_bwd_host_workspace_size(2, 2, 16, 64, 1, 2) == 0   # fp16 grads of bf16


@pytest.mark.parametrize("kw,want", [
    (dict(q=0), 1), (dict(dv=0), 1), (dict(workspace=0), 1),
    (dict(batch_chunk=0), 1),
    (dict(workspace_bytes=1024), 1),
    (dict(workspace=FAKE + 64), 1),        # not 256-byte aligned
    (dict(d=12), 1), (dict(d=136), 2),
    (dict(scale=float("nan")), 1),
    (dict(grad_dtype=2), 1),
])
def test_host_rejects_invalid_arguments(fake_lib, kw, want):
    from exact_attention_fwd_gb300 import _lib
    a = dict(q=FAKE, k=2 * FAKE, v=3 * FAKE, dO=4 * FAKE, o=5 * FAKE, lse=6 * FAKE, dq=7 * FAKE,
             dk=8 * FAKE, dv=9 * FAKE, B=4, H=2, N=16, d=64, scale=0.125, causal=1, dtype=1,
             grad_dtype=1, batch_chunk=2, workspace=16 * FAKE, workspace_bytes=1 << 24,
             stream=None)
    a.update(kw)
    assert _lib.fa_fwd_bwd_host(**a) == want


def test_unfused_workspace_size(lib):
    from exact_attention_fwd_gb300 import _lib
    # S (2 x 3 x 100 x 100 floats), O' (2 x 100 x 3 x 64 floats), l (2 x 3 x 100
    # floats), each rounded up to 256 bytes, then 32 MiB for the GEMMs
    assert _lib.fa_fwd_unfused_workspace_size(2, 3, 100, 64) == \
        240128 + 153600 + 2560 + (32 << 20)
    assert _lib.fa_fwd_unfused_workspace_size(0, 3, 100, 64) == 0


@pytest.mark.parametrize("kw,want", [
    (dict(q=0), 1), (dict(workspace=0), 1),
    (dict(workspace_bytes=1000), 1),
    (dict(workspace=16 * FAKE + 128), 1),   # not 256-byte aligned
    (dict(d=20), 1), (dict(d=136), 2),
    (dict(dtype=0), 2),                     # float32: not on this path
    (dict(q=FAKE + 4), 1),                  # misaligned
    (dict(scale=float("inf")), 1),
])
def test_unfused_rejects_invalid_arguments(fake_lib, kw, want):
    from exact_attention_fwd_gb300 import _lib
    a = dict(q=FAKE, k=2 * FAKE, v=3 * FAKE, o=4 * FAKE, lse=5 * FAKE, B=1, H=1, N=16, d=64,
             scale=0.125, causal=1, dtype=1, workspace=16 * FAKE, workspace_bytes=1 << 26,
             stream=None)
    a.update(kw)
    assert _lib.fa_fwd_unfused(**a) == want


def test_tf32x3_workspace_size(lib):
    from exact_attention_fwd_gb300 import _lib
    # 4 split copies of [1, 10, 2, 8] floats (640 -> 768 bytes each) and 2 of
    # V^T [1, 2, 8, 12] floats (768 bytes each)
    assert _lib.fa_fwd_tf32x3_workspace_size(1, 2, 10, 8) == 4 * 768 + 2 * 768
    assert _lib.fa_fwd_tf32x3_workspace_size(1, 2, 0, 8) == 0


@pytest.mark.parametrize("kw,want", [
    (dict(q=0), 1), (dict(workspace=0), 1),
    (dict(d=136), 2), (dict(d=12), 1),
    (dict(workspace_bytes=100), 1),
    (dict(workspace=16 * FAKE + 64), 1),
    (dict(o=FAKE), 1),                     # aliases q
    (dict(scale=float("nan")), 1),
])
def test_tf32x3_rejects_invalid_arguments(fake_lib, kw, want):
    from exact_attention_fwd_gb300 import _lib
    a = dict(q=FAKE, k=2 * FAKE, v=3 * FAKE, o=4 * FAKE, lse=5 * FAKE, B=1, H=1, N=16, d=64,
             scale=0.125, causal=1, workspace=16 * FAKE, workspace_bytes=1 << 22, stream=None)
    a.update(kw)
    assert _lib.fa_fwd_tf32x3(**a) == want


def test_missing_library_raises(monkeypatch, tmp_path):
    """No fallback: without libfa.so every binding raises instead of computing."""
    from exact_attention_fwd_gb300 import _lib
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "libfa.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    for call in (lambda: _lib.load(),
                 lambda: _lib.fa_bwd_workspace_size(1, 1, 128),
                 lambda: _lib.fa_fwd_tf32x3_workspace_size(1, 1, 128, 64),
                 lambda: _lib.fa_fwd_unfused_workspace_size(1, 1, 128, 64)):
        with pytest.raises(RuntimeError, match="not built"):
            call()


@pytest.mark.parametrize("kw,want", [
    (dict(q=0), 1), (dict(workspace=0), 1),
    (dict(d=72), 2),                       # the 3xTF32 backward takes d <= 64
    (dict(d=12), 1),
    (dict(workspace_bytes=100), 1),
    (dict(dq=FAKE), 1),                    # aliases q
    (dict(scale=float("nan")), 1),
])
def test_bwd_tf32x3_rejects_invalid_arguments(fake_lib, kw, want):
    from exact_attention_fwd_gb300 import _lib
    a = dict(q=FAKE, k=2 * FAKE, v=3 * FAKE, o=4 * FAKE, lse=5 * FAKE, dO=6 * FAKE,
             dq=8 * FAKE, dk=10 * FAKE, dv=12 * FAKE, B=1, H=1, N=16, d=64, scale=0.125,
             causal=1, workspace=16 * FAKE, workspace_bytes=1 << 24, stream=None)
    a.update(kw)
    assert _lib.fa_bwd_tf32x3(**a) == want
