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


def test_reference_arm_under_torchrun_prints_once_from_rank0():
    """Launched as the driver launches N > 1 (here 2 gloo ranks on the CPU): rank 0
    alone runs the oracle and prints; the other rank exits 0 without work."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
                        "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                        "--gpus", "2", "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "3", "--ref-sample-tokens", "8"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT,
                       env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.strip().splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["n_gpus"] == 2 and j["value"] > 0
