"""Register spills of the tcgen05 kernels, from ptxas (compile only, no GPU).

The hot-path instantiations must not spill.  The few variants with known small
spills are listed; any spill elsewhere fails, so a change to a shared loop that
tips a kernel's register split over is caught before it reaches a GPU.
"""
import os
import re
import subprocess

import pytest

from exact_attention_fwd_gb300 import build

SOURCES = ("tc_fwd.cu", "tc_bwd.cu", "tf32x3_fwd.cu", "tf32x3_bwd.cu")

# (kernel, template arguments as digits) with known, tolerated spills
#   fwd_tc_kernel<DP, causal, f16, split>, bwd_tc_kernel<DP, causal, dKdV, f32grad, f16>
KNOWN = [
    ("bwd_tc_kernel", r"64,0,1,[01],[01]"),     # non-causal dK/dV, DP = 64
    ("bwd_tc_kernel", r"128,[01],[01],[01],[01]"),  # every DP = 128 backward
]


def _compile_all(out):
    try:
        exe = build.nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    csrc = os.path.join(build.ROOT, "exact_attention_fwd_gb300", "csrc")
    procs = []
    for src in SOURCES:
        cmd = [exe, *build.ARCH, *build.NVCC_FLAGS, "-I" + csrc, "-Xptxas", "-v", "-c",
               os.path.join(csrc, src), "-o", os.path.join(out, src + ".o")]
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                            text=True)))
    reports = {}
    for src, p in procs:
        stdout, stderr = p.communicate(timeout=900)
        assert p.returncode == 0, f"nvcc failed on {src}:\n{stderr[-2000:]}"
        reports[src] = stdout + stderr
    return reports


def _kernel_name(mangled):
    """The `*_kernel` identifier of a mangled entry name (length-prefixed)."""
    for m in re.finditer(r"\d+", mangled):
        ident = mangled[m.end():m.end() + int(m.group())]
        if ident.endswith("_kernel") and re.fullmatch(r"[A-Za-z_]\w*", ident):
            return ident
    return mangled


def _spills(report):
    """(kernel name, template digits, spill store bytes, spill load bytes) per entry."""
    rows, cur = [], None
    for line in report.splitlines():
        m = re.search(r"Compiling entry function '(\S+)'", line)
        if m:
            cur = m.group(1)
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m and cur:
            args = ",".join(re.findall(r"(?:Li|Lb)(\d+)E", cur))
            rows.append((_kernel_name(cur), args, int(m.group(1)), int(m.group(2))))
            cur = None
    return rows


@pytest.fixture(scope="module")
def spill_rows(tmp_path_factory):
    rows = []
    for report in _compile_all(str(tmp_path_factory.mktemp("spills"))).values():
        rows.extend(_spills(report))
    return rows


def test_every_kernel_reported(spill_rows):
    names = {r[0] for r in spill_rows}
    for k in ("fwd_tc_kernel", "bwd_tc_kernel", "fwd_tf32x3_kernel", "bwd_tf32x3_kernel",
              "split_qk_kernel", "split_vt_kernel"):
        assert k in names
    # 16 forward and 32 backward instantiations; 3xTF32: 4 forward (DP, causal) and 4
    # backward (dK/dV, causal)
    assert sum(r[0] == "fwd_tc_kernel" for r in spill_rows) == 16
    assert sum(r[0] == "bwd_tc_kernel" for r in spill_rows) == 32
    assert sum(r[0] == "fwd_tf32x3_kernel" for r in spill_rows) == 4
    assert sum(r[0] == "bwd_tf32x3_kernel" for r in spill_rows) == 4


def test_hot_path_does_not_spill(spill_rows):
    hot = {("fwd_tc_kernel", "64,1,0,0"), ("fwd_tc_kernel", "128,1,0,0"),
           ("bwd_tc_kernel", "64,1,0,0,0"), ("bwd_tc_kernel", "64,1,1,0,0"),
           ("fwd_tf32x3_kernel", "64,1"), ("fwd_tf32x3_kernel", "64,0"),
           ("fwd_tf32x3_kernel", "128,1"), ("fwd_tf32x3_kernel", "128,0"),
           ("bwd_tf32x3_kernel", "0,1"), ("bwd_tf32x3_kernel", "1,1"),
           ("bwd_tf32x3_kernel", "0,0"), ("bwd_tf32x3_kernel", "1,0")}
    seen = set()
    for name, args, st, ld in spill_rows:
        if (name, args) in hot:
            seen.add((name, args))
            assert st == 0 and ld == 0, f"{name}<{args}> spills {st} / {ld} bytes"
    assert seen == hot


def test_spills_only_where_known(spill_rows):
    for name, args, st, ld in spill_rows:
        if st == 0 and ld == 0:
            continue
        assert any(name == k and re.fullmatch(pat, args) for k, pat in KNOWN), \
            f"new spill: {name}<{args}> {st} / {ld} bytes"
