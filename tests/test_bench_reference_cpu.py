"""bench.py's reference arm (the CPU oracle, timed on the host cores) prints one
JSON line in the benchmark's format, for the workload's own configuration."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "1", "--warmup", "3",
                        "--ref-sample-tokens", "16"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.strip().splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference"
    assert j["metric"] == "MoE layer fwd+bwd tokens/s" and j["unit"] == "tokens/s"
    assert j["higher_is_better"] is True and j["value"] > 0
    assert j["warmup"] >= 3 and j["steps"] == 1
    cfg = j["config"]
    assert cfg["workload"] == "tiny" and cfg["T"] == 256 and cfg["sample_tokens_per_step"] == 16
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["value"] == j["value"]
    assert j["cpu_baseline"]["cores"] >= 1
    assert j["e2e"] == {"value": j["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
