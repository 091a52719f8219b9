"""The reference arm of bench.py (the CPU oracle timed on the host cores) keeps the JSON line the
benchmark driver reads: run here on the CPU with a tiny step count, and once more with a time
budget small enough that every step becomes a token sample of the layers."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _check_line(line, steps, warmup):
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "impl", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["steps"] == steps and line["warmup"] == warmup
    assert line["unit"] == "GB/s" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["config"]["workload"] == "gqa_decode_mlx4g32"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


@pytest.mark.timeout(600)
def test_reference_arm_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                          "--warmup", "1"], capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, out.stdout
    line = json.loads(lines[0])
    _check_line(line, 2, 1)
    assert line["config"]["step"] == "the full 16-layer step"


@pytest.mark.timeout(600)
def test_reference_arm_samples_tokens_under_a_small_budget(capsys):
    sys.path.insert(0, ROOT)
    import argparse
    import bench
    bench.run_reference(argparse.Namespace(steps=40, warmup=2, gpus=1), budget_s=0.5)
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    line = json.loads(lines[-1])
    _check_line(line, 40, 2)
    step = line["config"]["step"]
    assert "sample" in step, step
    n_tok = int(step.split("a ")[1].split("-token")[0])
    assert 256 <= n_tok < 8192 and n_tok % 16 == 0
