"""The JSON line of bench.py's reference arm (the CPU oracle, timed on a row
sample of the workload): one line with the keys and units the GPU arm uses,
only rank 0 printing under a multi-rank launch, and the warm-up floor."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

CMD = [sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--reference-rows", "8"]


def _run(args, env=None):
    return subprocess.run(CMD + args, cwd=ROOT, env=dict(os.environ, **(env or {})), capture_output=True, text=True,
                          timeout=600)


def test_reference_arm_prints_one_complete_line():
    r = _run(["--steps", "2", "--warmup", "3"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC
    assert d["unit"] == "ms" and d["higher_is_better"] is False
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["scaling"] == "weak" and d["data"] == "synthetic" and d["vs_baseline"] is None
    assert d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == "ms" and cb["cores"] >= 1
    assert "rows" in cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == "ms"
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    r = _run(["--steps", "1", "--warmup", "3"], env={"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_fewer_than_three_warmup_steps_are_refused():
    r = _run(["--steps", "1", "--warmup", "2"])
    assert r.returncode != 0
