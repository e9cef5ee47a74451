"""bench.py keeps its one-line JSON contract on a GPU: a short run of the
headline step (no extras) prints one line whose keys, units and internal
arithmetic agree (value = offsets x steps / time, roofline.frac =
achieved / peak, one launch of the library's kernel per step)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_contract():
    r = subprocess.run([sys.executable, "bench.py", "--steps", "30", "--warmup", "3",
                        "--extras", "0"], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "gpu_launches", "clocks", "roofline"):
        assert key in d, key
    assert d["unit"] == "offsets/s" and d["higher_is_better"] is True
    assert d["steps"] == 30 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["gpu_launches"] == 30
    offsets = d["config"]["offsets"]
    assert d["value"] == pytest.approx(offsets / (d["ms_per_step"] * 1e-3), rel=1e-6)
    rf = d["roofline"]
    assert rf["bound"] == "alu" and rf["unit"] == "Tdp4a/s"
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"], rel=1e-9)
    assert 0.05 < rf["frac"] < 1.2
    # achieved = algorithmic dp4a per launch / mean launch time
    per = int(rf["algorithmic_per_unit"].split()[0])
    assert per == 1024                     # 64x64 template, box form: one dp4a per 4 pixels
    assert rf["achieved"] * 1e12 == pytest.approx(
        offsets * per / (d["ms_per_step"] * 1e-3), rel=1e-6)
