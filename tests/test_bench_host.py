"""bench.py's host logic on the CPU: the reference (oracle) arm's JSON line, the workload
override used for smaller profiling cases, and the oracle shards of the CPU baseline."""
import argparse
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "0", "--steps", "2", "--warmup", "1"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT, check=True).stdout
    lines = [ln for ln in out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["unit"] == bench.UNIT and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "tiny_B4_K8_nx16_C32"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_workload_override_renames_after_its_sizes():
    args = argparse.Namespace(workload=4, batch=1024, seq=32)
    w = bench.workload(args)
    assert (w.B, w.K, w.n_x, w.C) == (1024, 32, 64, 256)
    assert w.name == "stress_B1024_K32_nx64_C256"
    assert bench.workload_tag(w) == "stress_B1024_K32"
    plain = bench.workload(argparse.Namespace(workload=1, batch=None, seq=None))
    assert plain.name == "pages_B32_K64_nx48_C128"
    assert bench.workload_tag(plain) == "pages_B32_K64"


@pytest.mark.parametrize("r0,r1", [(0, 4), (1, 3)])
def test_oracle_shard_counts_its_rows(r0, r1):
    from recurrent_cfc_cell_gb300 import inputs

    w = inputs.CONFIGS[0]
    units, dt = bench._oracle_shard(w, r0, r1, 0.05)
    assert dt >= 0.05
    assert units > 0 and units % ((r1 - r0) * w.K) == 0
