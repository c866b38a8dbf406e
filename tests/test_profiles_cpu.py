"""The committed ncu traffic summary (profiles/dram_traffic.json) agrees with
the workloads it was taken on: every entry's algorithmic bytes equal the bytes
recomputed here from the seeded workload metadata (every cached K and V row of
every KV head once; MLA: every latent row once; cache writes: rows read plus
rows and scales written), read + write add up to the stated traffic, and a
decode kernel's measured DRAM reads are not below its algorithmic bytes (a
capture that saw less than the step reads was not of the full workload).  CPU
only; no GPU figure is recomputed."""
import json
import os

import numpy as np
import pytest

from paged_kv_decode_06_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
    TRAFFIC = json.load(f)


def _algorithmic(name):
    if name.startswith("cache_write_T"):
        T, kind = name[len("cache_write_T"):].split("_", 1)
        T, Hkv, D = int(T), 8, 128
        esz = 2 if kind == "bf16" else 1
        return T * Hkv * D * 2 * (2 + esz) + (T * Hkv * 2 * 4 if kind.endswith("per_token") else 0)
    if name in wl.MLA_CONFIGS:
        spec = wl.MLA_CONFIGS[name]
        sl = wl.draw_metadata(spec, np.random.default_rng(spec.seed))[0]
        return int(sl.astype(np.int64).sum()) * spec.head_dim * (1 if spec.kv_dtype == "fp8" else 2)
    spec = wl.CONFIGS[name]
    sl = wl.draw_metadata(spec, np.random.default_rng(spec.seed))[0]
    per_row = spec.head_dim * (1 if spec.kv_dtype == "fp8" else 2) + (4 if spec.token_scale_range is not None else 0)
    return int(sl.astype(np.int64).sum()) * spec.num_kv_heads * 2 * per_row


@pytest.mark.parametrize("name", sorted(TRAFFIC))
def test_traffic_entry_matches_its_workload(name):
    e = TRAFFIC[name]
    assert e["algorithmic_bytes"] == _algorithmic(name)
    assert e["dram_bytes_per_launch"] == e["dram_bytes_read"] + e["dram_bytes_write"]
    assert len(e["kernel_source_sha256"]) == 64 and e["source"].startswith("ncu ")
    if not name.startswith("cache_write_T"):
        assert e["dram_bytes_read"] >= e["algorithmic_bytes"]


def test_every_benchmarked_workload_has_an_entry():
    assert set(TRAFFIC) >= {"llama3_8b", "fp8", "mtp", "batch1_32k", "verify8", "fp8_pertoken", "mla_tp8",
                            "mla_mtp_fp8"}
