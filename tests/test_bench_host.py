"""Host-side logic of bench.py, on CPU: FLOP and byte accounting, clock parsing,
the max-over-ranks reduction across two gloo ranks, and the reference arm."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_flop_accounting():
    fwd, bwd = bench.flops_step(64, 16, 1024, 64, True)
    assert fwd == pytest.approx(137.438953472e9)       # 4 B H N^2 d / 2
    assert bwd == pytest.approx(2.5 * fwd)
    w = bench.kernel_work(64, 16, 1024, 64, True)
    assert w["fwd_tc_kernel"] == ("tensor", fwd)
    assert w["bwd_dq"][1] + w["bwd_dkdv"][1] == pytest.approx(3.5 * fwd)
    assert w["dot_do_o_kernel"] == ("hbm", 2 * 64 * 16 * 1024 * 64 * 2 + 4 * 64 * 16 * 1024)


def test_parse_clocks():
    lines = [
        "0, 1900, 2070, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1800, 2070, 1300.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 1850, 2070, 1200.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage",
    ]
    c = bench.parse_clocks(lines)
    assert c["sm_mhz"] == 1850 and c["sm_max_mhz"] == 2070 and c["samples"] == 3
    assert c["reasons"] == ["sw_power_cap"]
    assert bench.parse_clocks([])["sm_mhz"] is None


def test_aggregate_uses_slowest_rank():
    assert bench.aggregate([10.0, 10.0], [1.0, 2.0]) == 10.0


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


WORKER = r"""
import os, sys
sys.path.insert(0, {root!r})
import bench
dist = bench.init_dist(2, False)
r = int(os.environ["RANK"])
t = bench.max_over_ranks(1.5 + r, dist)
print("RESULT", r, t, bench.aggregate([100.0, 100.0], [t, t]))
dist.destroy_process_group()
"""


def test_max_over_ranks_two_gloo_ranks():
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER.format(root=ROOT)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (out, err) in zip(procs, outs):
        assert p.returncode == 0, err
        line = [ln for ln in out.splitlines() if ln.startswith("RESULT")][0].split()
        assert float(line[2]) == 2.5                      # max over ranks
        assert float(line[3]) == pytest.approx(200.0 / 2.5)


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "3"], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["unit"] == "TFLOP/s" and j["value"] > 0
    assert j["metric"] == bench.METRIC
    assert j["e2e"]["h2d_bytes_per_step"] == 0 and j["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "2", "--warmup", "3"], capture_output=True,
                       text=True, timeout=120, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""
