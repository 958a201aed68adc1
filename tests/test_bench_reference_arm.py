"""bench.py's reference arm (the fp64 oracle on the host cores) on CPU: one
step prints one JSON line with the keys of the bench contract, and its
config names the workload with the same string the GPU arm prints."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 0
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}

    sys.path.insert(0, ROOT)
    try:
        import bench
        from delta_rule_linear_dpfp_gb300 import inputs
        assert d["config"]["workload"] == bench.workload_name(inputs.FORWARD_CONFIGS[bench.WORKLOAD])
        assert d["metric"] == bench.METRIC
    finally:
        sys.path.remove(ROOT)


def test_reference_arm_under_torchrun_prints_once():
    """Launched as a run on N > 1 GPUs is launched (torchrun, two ranks): rank 0
    alone runs the oracle and prints the line, the other rank exits 0."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
                        "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0


def test_recorded_traffic_belongs_to_the_current_sources():
    """The DRAM traffic bench.py reports for the headline kernel comes from an
    ncu capture tied to a hash of the forward's sources; any change to them
    (a comment included) needs a new capture, else the line reports null."""
    sys.path.insert(0, ROOT)
    try:
        import bench
        rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
        entry = rec[f"chunk_fused_kernel@{bench.WORKLOAD}"]
        assert entry["source_hash"] == bench.source_hash(bench.FORWARD_SOURCES)
        assert entry["dram_bytes_per_launch"] == entry["read"] + entry["write"] > 0
    finally:
        sys.path.remove(ROOT)
