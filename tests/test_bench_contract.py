"""bench.py's one-line JSON contract, checked on the CPU through its reference
arm (the oracle timed on host cores), on the tiny workload."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          capture_output=True, text=True, timeout=300)


def test_reference_arm_prints_one_contract_line():
    r = _run("--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "impl"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["higher_is_better"] is True and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["config"]["workload"].startswith("tiny")
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # tokens/s and ms per step describe the same timing; the tiny step fits
    # its budget, so each timed step is the whole workload
    assert d["reference_step"] == "the whole workload per step"
    assert d["sampled_tokens_per_step"] == d["config"]["tokens_per_step"]
    assert abs(d["value"] * d["ms_per_step"] * 1e-3 - d["sampled_tokens_per_step"]) < 1e-6 * d["value"]
    # the same config object as the GPU arm's line
    for key in ("workload", "num_seqs", "tokens_per_step", "computed_query_rows", "kv_bytes_read", "l2",
                "parallelism"):
        assert key in d["config"], key


def test_fewer_than_three_warmup_steps_are_refused():
    r = _run("--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "2")
    assert r.returncode != 0
    assert "warmup" in r.stderr
