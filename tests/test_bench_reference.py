"""bench.py's reference arm (the oracle timed on the host cores) prints one JSON
line with the keys the harness reads, for a decode workload; for a workload
the oracle baseline does not cover it prints an ``unavailable`` line.  CPU
only: the reference arm never touches the GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        *args], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_reference_line_for_a_decode_workload():
    line = _run("--workload", "tiny", "--steps", "2", "--warmup", "3", "--ref-seconds", "0.2")
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["config"]["workload"] == "tiny" and line["config"]["num_seqs"] == 4
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert "of tiny" in line["cpu_baseline"]["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"],
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_line_unavailable_for_prefill():
    line = _run("--workload", "prefill", "--steps", "1", "--warmup", "3")
    assert line["impl"] == "reference" and "unavailable" in line
