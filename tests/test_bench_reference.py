"""The benchmark's reference arm (``bench.py --impl reference``: the CPU fp64
oracle timed on the host cores) runs on a machine without a GPU and prints
one JSON line with the keys the benchmark contract names."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
           "--warmup", "1", "--workload", "blockdiag_b1h2n256d128_bs64_f16", "--threads", "2"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["cores"] == 2 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["config"]["workload"] == "blockdiag_b1h2n256d128_bs64_f16"
    # the flop count of one head: 4 * D * L * bs attended pairs
    assert abs(d["value"] - 4 * 128 * 256 * 64 / (d["ms_per_step"] * 1e-3) / 1e12) <= 1e-6 * d["value"]
