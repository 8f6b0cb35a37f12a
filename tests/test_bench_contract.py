"""bench.py's reference arm (no GPU): the oracle timed on the host cores prints
one JSON line with the contract's keys, and fewer than 3 warm-up steps are
refused."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          capture_output=True, text=True, timeout=300)


def test_reference_arm_prints_one_contract_line():
    r = _bench("--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 3 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny_gqa2_d64_f32"
    # the same config keys as the GPU arm prints (bench_config), so the two lines compare
    import bench
    assert d["config"] == json.loads(json.dumps(bench.bench_config(
        __import__("paged_kv_cache_215_gb300.workloads", fromlist=["x"]).FULL["tiny"](), 1)))
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_fewer_than_three_warmup_steps_are_refused():
    r = _bench("--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "2")
    assert r.returncode != 0 and "warmup" in r.stderr


def test_reference_arm_under_torchrun_prints_once():
    """Launched the way a multi-GPU run launches it (one process per rank),
    rank 0 alone prints the line; the other ranks exit 0 without work."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1", "--master-port",
                        str(port), os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--gpus", "2", "--steps", "3", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    assert json.loads(lines[0])["impl"] == "reference"
