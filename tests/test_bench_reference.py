"""bench.py's reference arm (the float64 oracle on the host cores) on the
CPU: one JSON line with the contract's keys on rank 0, nothing and exit 0 on
the other ranks, and the warm-up floor enforced."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ARGS = ["--impl", "reference", "--workload", "layer1", "--steps", "3", "--warmup", "3"]


def _bench(args, **env):
    e = dict(os.environ, **env)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=e,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_contract_line():
    p = _bench(ARGS)
    assert p.returncode == 0, p.stderr[-800:]
    lines = [x for x in p.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == "MoE-layer decode tokens/s (one layer)" and d["unit"] == "tok/s"
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["vs_baseline"] is None and d["data"] == "synthetic" and d["dtype"] == "f64"
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert 1 <= cb["cores"] <= 6  # the six steps spread over at most six processes
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # value = tokens per second over the processes that ran: cores x 1 token / seconds per step
    assert abs(d["value"] - cb["cores"] * 1e3 / d["ms_per_step"]) <= 1e-3 * d["value"]


def test_reference_arm_is_silent_on_other_ranks():
    p = _bench(ARGS, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    assert p.returncode == 0, p.stderr[-800:]
    assert p.stdout.strip() == ""


def test_fewer_than_three_warmup_steps_are_rejected():
    p = _bench(["--impl", "reference", "--workload", "layer1", "--steps", "3", "--warmup", "2"])
    assert p.returncode == 2
    assert "--warmup must be >= 3" in p.stderr
