"""bench.py's reference arm (the oracle timed on the host cores) on the CPU: one
JSON line with the metric, unit and direction of the GPU arm and the keys the
measurement contract asks for; under torchrun only rank 0 runs it."""

import json
import os
import subprocess
import sys

from conftest import ROOT


def _run(args, env_extra=None):
    env = dict(os.environ, **(env_extra or {}))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          cwd=ROOT, env=env, timeout=600)


def test_reference_arm_prints_one_contract_line():
    res = _run(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, res.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "rows/s" and d["higher_is_better"] is True
    assert d["metric"].startswith("verified logit rows/sec")
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] >= 3 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "ragged_mixed_b128_v262144"  # the largest single-GPU workload
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_runs_on_rank_zero_only():
    res = _run(["--impl", "reference", "--steps", "1", "--warmup", "3"],
               {"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2", "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": "29571"})
    assert res.returncode == 0, res.stderr[-2000:]
    assert not [l for l in res.stdout.splitlines() if l.strip().startswith("{")], res.stdout
