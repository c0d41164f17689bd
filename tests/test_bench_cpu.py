"""The benchmark's JSON-line contract, checked on its CPU arm (the oracle timed
on a bounded sample) at the smallest workload."""
import json
import os
import subprocess
import sys

import bench
from h3inputs import CONFIGS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "tiny",
                        "--steps", "2", "--warmup", "1"], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    # at least three untimed warm-up steps are run (and reported) whatever is asked
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["config"] == bench._config(CONFIGS["tiny"])
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]


def test_l2_note_follows_the_working_set():
    assert bench._config(CONFIGS["full"])["l2"].startswith("inputs larger than L2")
    assert bench._config(CONFIGS["medium"])["l2"].startswith("inputs larger than L2")
    assert "fits in the 129 MB L2" in bench._config(CONFIGS["small"])["l2"]
