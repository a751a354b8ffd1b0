"""The benchmark's host-side contract, on CPU: the reference arm's JSON line
(the oracle on bounded samples of the workload), the rank rule for N > 1,
and the FLOP count the TFLOP/s figures divide by."""
import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_flop_count_of_the_workload():
    # 10 B H S^2 d for the full mask (five 2 x S x S x d products), half causal
    full = 10.0 * 2 * 16 * 8192 * 8192 * 128
    assert bench.flops("full") == full
    assert bench.flops("causal") == full / 2
    assert bench.workload_name() == "attn_bwd_b2h16s8192d128_causal+full"


def test_reference_arm_other_ranks_do_no_work():
    class Args:
        steps, warmup = 1, 3
    assert bench.run_reference(Args(), rank=1) is None


def test_reference_arm_json_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    out = json.loads(lines[0])
    assert out["impl"] == "reference"
    assert out["metric"] == bench.METRIC and out["unit"] == "TFLOP/s"
    assert out["higher_is_better"] is True and out["steps"] == 1 and out["warmup"] == 3
    assert out["config"]["workload"] == bench.workload_name()
    assert out["value"] > 0
    cb = out["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == out["value"]
    assert "rows" in cb["sample"]
    e2e = out["e2e"]
    assert e2e["value"] == out["value"] and e2e["unit"] == out["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
