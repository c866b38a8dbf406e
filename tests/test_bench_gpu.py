"""The benchmark's JSON line on small workloads (a GPU run of bench.py): the
contract's keys, a clean device status, and end-to-end steps whose copied-back
results equal the direct call's."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("config", ["tiny", "mla_tiny"])
def test_bench_line_on_a_small_workload(config):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--config", config, "--steps", "24", "--warmup", "3",
           "--no-cpu-baseline", "--no-per-config", "--min-seconds", "0"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["steps"] == 24 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["device_status"] == 0
    assert d["value"] > 0 and d["roofline"]["bound"] == "hbm" and d["roofline"]["achieved"] > 0
    e = d["e2e"]
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert e["verified_steps"] >= 2 and e["verified_equal_to_direct_call"] is True
    assert e["value"] == max(e["pipelined_value"], e["serial_value"])
