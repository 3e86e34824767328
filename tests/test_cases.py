"""The named single-GPU workloads used to time and profile the entry points."""
import ast
import os

import pytest

from exact_attention_fwd_gb300 import cases

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_case_registry_matches_documented_names():
    assert sorted(cases.CASES) == ["bert_bwd", "bert_fwd", "gpt2_unfused", "long4_bwd",
                                   "long4_fwd", "long_fwd", "splitkv", "tf32x3", "tf32x3_bwd"]
    doc = cases.__doc__
    for name in cases.CASES:
        assert f"``{name}``" in doc
        assert callable(cases.CASES[name])


def test_cases_module_does_not_use_the_oracle():
    src = open(os.path.join(ROOT, "exact_attention_fwd_gb300", "cases.py")).read()
    for node in ast.walk(ast.parse(src)):
        if isinstance(node, ast.Import):
            assert all("oracle" not in a.name for a in node.names)
        if isinstance(node, ast.ImportFrom):
            assert "oracle" not in (node.module or "")


def test_profile_commands_name_committed_files():
    """Every capture summary gives a command that runs bench.py or the cases module."""
    pdir = os.path.join(ROOT, "profiles")
    for f in sorted(os.listdir(pdir)):
        if not f.endswith(".md"):
            continue
        text = open(os.path.join(pdir, f)).read()
        assert "<script>" not in text, f
        assert "_work" not in text, f
        assert ("python bench.py" in text or "exact_attention_fwd_gb300.cases" in text), f


@pytest.mark.gpu
@pytest.mark.parametrize("name", sorted(cases.CASES))
def test_case_runs(name):
    (B, H, N, d), ms, tflops = cases.run_case(name, reps=1)
    assert B >= 1 and H >= 1 and N >= 1 and d >= 1
    assert ms > 0.0 and tflops > 0.0
