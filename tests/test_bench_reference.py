"""The reference arm of bench.py on CPU (it times the oracle): the JSON line's
contract, and that under several ranks only rank 0 runs and prints."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CMD = [sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_exhaustive",
       "--steps", "2", "--warmup", "1"]


def _run(extra_env):
    env = dict(os.environ, **extra_env)
    return subprocess.run(CMD, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)


def test_reference_line_contract():
    p = _run({"RANK": "0", "WORLD_SIZE": "1"})
    assert p.returncode == 0, p.stderr[-2000:]
    line = json.loads(p.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["metric"] == "draft+verify cycles/s" and line["unit"] == "cycles/s"
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["n_gpus"] == 1 and line["steps"] == 2 and line["warmup"] == 1
    assert line["config"]["workload"] == "tiny_exhaustive"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == line["value"]
    assert cb["nproc"] >= 1 and cb["cpu_model"]
    # each timed step is one whole cycle: the rate and the step time agree
    assert abs(line["value"] * line["ms_per_step"] - 1000.0) < 1e-6 * 1000.0
    import bench
    w = bench.inputs.workload("tiny_exhaustive")
    assert line["config"] == bench.workload_config(w, 1)
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_other_ranks_exit_quietly():
    p = _run({"RANK": "1", "WORLD_SIZE": "2"})
    assert p.returncode == 0, p.stderr[-2000:]
    assert p.stdout.strip() == ""
