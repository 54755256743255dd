"""bench.py end to end on the GPU, briefly: one JSON line with the keys its readers use,
figures in range, and the per-config CPU baseline left out at this size (the full run
times it; here the CPU legs are switched off to keep the test short)."""
import json
import os
import subprocess
import sys

import pytest

from conftest import ROOT

pytestmark = pytest.mark.gpu


def test_bench_prints_one_line_with_the_metric_and_its_evidence(tmp_path):
    detail = tmp_path / "detail.json"
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "4", "--warmup", "3",
                          "--no-e2e", "--no-cpu-baseline", "--detail", str(detail)],
                         capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "quantize_amax_gbs", "quantize_amax_frac", "scale_update_us",
              "scale_update_launches", "roofline", "rows", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["steps"] == 4 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["gpu_launches"] == 4 * 4 and d["scale_update_launches"] == 1
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    # a streaming kernel cannot beat the copy peak by much, nor should it fall far below it
    assert 0.5 < r["frac"] < 1.2 and 0.5 < d["quantize_amax_frac"] < 1.2
    assert 0 < d["scale_update_us"] < 20
    if d.get("graph_node_floor_us") is not None:   # a one-element fill in the update's place
        assert 0 < d["graph_node_floor_us"] < d["scale_update_us"]
    for k, v in d["rows"].items():
        assert v > 0, k
    assert 0.5 < d["value"] / r["peak"] < 1.3      # the whole step, GB/s against the same peak
    assert json.loads(detail.read_text())["kernels"]["quantize_amax"]["us"] > 0
