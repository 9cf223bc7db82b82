"""bench.py on CPU: the reference arm's JSON line (the oracle timed on full
steps), the --gpus contract and the byte accounting of the two schedules."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3",
                        "--layers", "1"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    line = json.loads(lines[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["unit"] == "tokens/s" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"].startswith("C2")
    # measured on whole steps with the requested warm-up, not scaled from a sample
    assert line["steps"] == 2 and line["warmup"] == 3
    assert "scaled" not in line["cpu_baseline"]["sample"]


def test_more_gpus_need_one_process_each():
    r = subprocess.run([sys.executable, "bench.py", "--gpus", "2", "--steps", "1", "--warmup", "3"], cwd=ROOT,
                       capture_output=True, text=True, timeout=120, env={**os.environ, "WORLD_SIZE": "1"})
    assert r.returncode != 0 and "one process per GPU" in r.stderr


def test_deferred_schedule_saves_one_state_read_per_folded_item():
    """The deferred schedule folds inside the verify: per folded (layer,
    request, head) the state is read once for both, so a step moves
    4 V K bytes less per folded item than verify-then-commit."""
    sys.path.insert(0, ROOT)
    import bench
    from workloads import CONFIGS, draw_metadata
    cfg = CONFIGS["C2"]
    meta = draw_metadata(cfg, np.random.default_rng(5))
    acct = bench.step_accounting(cfg, meta)
    lens = np.minimum(np.diff(meta.query_start_loc), cfg.Q)
    acc = np.minimum(np.maximum(meta.num_accepted, 0), lens)
    folded = int(((meta.state_indices > 0) & (acc > 0)).sum())
    assert folded > 0
    assert acct["commit_items"] == cfg.L * cfg.H * folded
    assert acct["deferred_step_bytes"] == acct["step_bytes"] - cfg.L * cfg.H * folded * 4 * cfg.V * cfg.K
