"""CPU: bench.py's reference arm, the oracle timed on the host cores, prints one JSON line with
the benchmark contract's keys, on the GPU arm's metric, unit and workload; the swap path, which
has no arithmetic for the oracle to time, prints an `unavailable` line.  Both exit 0."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *args],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [line for line in out.stdout.splitlines() if line.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def test_reference_arm_json_line():
    sys.path.insert(0, ROOT)
    import bench

    # the headline workload is the largest one; the line for a smaller one has the same form
    assert bench.DEFAULT_WORKLOAD == "mha_b256_append" and bench.DEFAULT_WORKLOAD in bench.PER_CONFIG
    d = _run("--workload", "gqa4_b64", "--steps", "1", "--warmup", "3", "--ref-seqs-per-step", "2")
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 1 and d["warmup"] == 3
    assert d["config"]["workload"].startswith("gqa4_b64")
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_arm_swap_is_unavailable():
    d = _run("--path", "swap", "--steps", "1", "--warmup", "3")
    assert d["impl"] == "reference" and d["unavailable"]
