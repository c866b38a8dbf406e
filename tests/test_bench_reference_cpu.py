"""bench.py's reference arm (the float64 oracle timed on the host cores) keeps
the benchmark contract: one JSON line with impl "reference", the arm's metric
and step counts, a cpu_baseline describing the run, an e2e object without host
copies, and a run time bounded by --ref-total however many steps are asked for
(each step one bounded sample).  CPU only."""
import json
import os
import subprocess
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("config", ["tiny", "mla_tiny"])
def test_reference_arm_line(config):
    t0 = time.time()
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", config,
                        "--steps", "400", "--warmup", "3", "--ref-total", "4"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["steps"] == 400 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True and "metric" in d
    assert d["config"]["workload"] == config
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and "400 timed samples" in cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert time.time() - t0 < 240
