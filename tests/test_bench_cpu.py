"""bench.py on the host: the reference arm (the oracle on CPU cores) prints one JSON line with
the contract's keys, and the launch count claimed per step follows the call structure."""
import json
import os
import subprocess
import sys

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "3", "--warmup", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "dtype", "data", "config"):
        assert key in d, key
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 3
    # a step is one whole batch cycle: the step time and the cycle rate agree
    assert abs(d["ms_per_step"] * d["value"] / 1e3 - 1.0) < 1e-6
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]


def test_launches_per_step_follow_the_calls():
    sys.path.insert(0, ROOT)
    import bench
    # fusion 4 launches up to 256 new rows (the K/V epilogue kernel), else 3; attention 3 per layer; verify 2
    assert bench.launches_per_step(256, 5) == 4 + 15 + 2
    assert bench.launches_per_step(257, 5) == 3 + 15 + 2
    assert bench.launches_per_step(8, 1) == 4 + 3 + 2
