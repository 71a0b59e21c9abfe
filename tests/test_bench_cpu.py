"""The benchmark's CPU legs, on the tiny workload: the oracle sample behind `cpu_baseline`
and the `--impl reference` arm (one JSON line, rank 0)."""
import json
import os
import subprocess
import sys

import bench
import oscar_synthetic as syn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_oracle_sample_all_cores_and_one_core():
    r = bench.oracle_sample(syn.WORKLOADS["tiny_gqa4_1k"], 0.4)
    assert r["kind"] == "oracle" and r["unit"] == "tokens/s"
    assert r["cores"] >= 1
    assert r["value"] > 0 and r["single_core_value"] > 0
    assert f"on {r['cores']} host cores" in r["sample"]


def test_reference_arm_prints_one_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny_gqa4_1k", "--steps", "2", "--warmup", "3", "--cpu-seconds", "0.6"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] == d["cpu_baseline"]["value"] == d["e2e"]["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["higher_is_better"] is True and d["unit"] == "tokens/s"
