"""The benchmark's reference arm (the fp64 oracle on the host cores) launched
the way a two-rank run launches it: one process per rank under
torch.distributed.run over gloo.  Rank 0 alone prints one JSON line with the
contract's keys; the other rank exits 0 without work."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_reference_arm_two_ranks_prints_one_line():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--cpu-tokens", "1024"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 1 and d["warmup"] == 3
    assert d["metric"] == "attention fwd+bwd TFLOP/s (bf16)" and d["unit"] == "TFLOP/s"
    assert d["higher_is_better"] is True and d["value"] > 0
    assert d["config"]["workload"] == "longctx_b1h16n16384d128"
    assert d["config"]["parallelism"] == "replicas" and d["config"]["l2"] == "flushed between steps"
    cpu = d["cpu_baseline"]
    assert "first 1024 tokens" in cpu["sample"]
    assert cpu["kind"] == "oracle" and cpu["value"] == d["value"] and cpu["cores"] >= 1 and cpu["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
