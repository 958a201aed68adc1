"""bench.py's own arm on the GPU: a short run prints one JSON line with the
keys of the bench contract (clocks, the roofline with its recorded traffic,
the end-to-end figure with its copies, the launch count) and the same
workload string as the reference arm."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_keys():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    steps = 40
    r = subprocess.run([sys.executable, "bench.py", "--steps", str(steps), "--warmup", "3", "--no-rows", "--no-cpu"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["steps"] == steps and d["warmup"] == 3
    assert d["n_gpus"] == 1 and d["dtype"] == "bf16" and d["data"] == "synthetic" and d["vs_baseline"] is None
    roof = d["roofline"]
    assert roof["bound"] in ("hbm", "tensor", "alu") and roof["peak"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-9
    assert roof["traffic"] is None or roof["traffic"] > 0
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] >= steps
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]

    sys.path.insert(0, ROOT)
    try:
        import bench
        from delta_rule_linear_dpfp_gb300 import inputs
        assert d["config"]["workload"] == bench.workload_name(inputs.FORWARD_CONFIGS[bench.WORKLOAD])
        assert d["metric"] == bench.METRIC
    finally:
        sys.path.remove(ROOT)
