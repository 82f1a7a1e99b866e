"""bench.py's reference arm on the CPU: the oracle timed on host cores, printed as one JSON line with
the keys of the GPU arm's line (impl, metric, value, unit, steps, warmup, ms_per_step, config,
cpu_baseline, e2e with zero copy bytes).  Under a launcher that starts several ranks, rank 0
alone prints it and the other ranks exit without work."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra):
    env = dict(os.environ)
    env.update(env_extra)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return [ln for ln in r.stdout.splitlines() if ln.strip()]


def test_reference_arm_prints_one_line_with_the_contract_keys():
    lines = _run({"RANK": "0", "WORLD_SIZE": "1"})
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["unit"] == "GB/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 2 and d["warmup"] == 3 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == "llama7b_decode_4bit_g128"
    assert d["config"]["M"] == 1 and d["config"]["K"] == 4096 and d["config"]["N"] == 11008
    assert 32 <= d["config"]["sample_columns"] <= 11008 and d["config"]["sample_columns"] % 32 == 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == d["value"] and cb["sample"]
    assert cb["host"]["nproc"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["vs_baseline"] is None


def test_reference_arm_other_ranks_exit_without_work():
    assert _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}) == []
