"""The bench's reference arm (the float64 oracle timed on the host cores) keeps the JSON contract the
driver reads: one line with impl, metric, value, unit, steps, warmup, ms_per_step, higher_is_better,
dtype, config, cpu_baseline and an e2e entry with no host-device traffic.  Host only (no GPU)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3",
                          "--ref-positions", "256"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "dtype",
              "config", "cpu_baseline", "e2e"):
        assert k in j, k
    assert j["steps"] == 1 and j["warmup"] == 3 and j["higher_is_better"] is True
    assert j["value"] > 0 and j["ms_per_step"] > 0
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["cores"] >= 1
    assert j["cpu_baseline"]["host_cores"] >= j["cpu_baseline"]["cores"] // 2
    assert j["e2e"]["h2d_bytes_per_step"] == 0 and j["e2e"]["d2h_bytes_per_step"] == 0
    assert j["e2e"]["value"] == j["value"]
    assert j["config"]["workload"] == "sweep_bf16_B1H8N131072K256"
