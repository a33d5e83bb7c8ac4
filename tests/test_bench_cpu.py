"""The bench's reference arm (the fp64 oracle timed on host cores) and its
JSON line, on the CPU: the line carries the fields every bench line carries,
and ranks other than 0 print nothing and exit 0."""
from __future__ import annotations

import json
import os
import subprocess
import sys
from pathlib import Path

ROOT = Path(__file__).resolve().parents[1]


def _run(extra_env=None, *args):
    env = dict(os.environ)
    env.update(extra_env or {})
    return subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference", "--workload", "tiny",
                           "--steps", "4", "--warmup", "3", *args],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)


def test_reference_arm_prints_one_contract_line():
    r = _run()
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["unit"] == "ms/token" and d["higher_is_better"] is False
    assert d["value"] > 0 and d["ms_per_step"] == d["value"]
    assert d["steps"] == 4 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "tiny" and d["config"]["ctx_last_timed"] - d["config"]["ctx_first_timed"] == 3
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "ms/token", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_do_no_work():
    r = _run({"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
