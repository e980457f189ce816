"""bench.py's reference arm on the CPU: `--impl reference` times the oracle
on the host cores and prints one JSON line with the keys of the bench
contract (metric, value, unit, steps, warmup, cpu_baseline, e2e with no
host-device bytes); under torchrun only rank 0 runs it, the other ranks exit
0 without work."""
import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(extra_env):
    env = dict(os.environ, **extra_env)
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--config", "tiny", "--steps", "2", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return [json.loads(line) for line in r.stdout.splitlines() if line.startswith("{")]


def test_reference_line():
    lines = _run({"RANK": "0"})
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 1 and d["value"] > 0 and d["ms_per_step"] > 0
    assert d["dtype"] == "f64" and d["data"] == "synthetic" and d["vs_baseline"] is None
    assert d["config"]["seq_len"] == 256 and d["config"]["sample_tokens"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_other_ranks_do_nothing():
    assert _run({"RANK": "1", "WORLD_SIZE": "2"}) == []
