"""The benchmark's contract line on the GPU: one short native run of bench.py prints one
JSON line whose keys, units and arithmetic are the ones the line promises (roofline =
algorithmic bytes over the mean launch time against the peak, tokens/s = rows over the
step time, the e2e byte counts of the copies, the per-workload summary at its end)."""
import json
import subprocess
import sys

import pytest

from conftest import ROOT

pytestmark = pytest.mark.gpu


def test_native_line_keeps_the_contract():
    r = subprocess.run([sys.executable, "bench.py", "--steps", "20", "--warmup", "3",
                        "--e2e-steps", "20", "--variant-steps", "20"],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-4000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, "exactly one line on stdout"
    line = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "clocks", "gpu_launches", "configs"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["steps"] == 20 and line["warmup"] == 3
    assert line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["config"]["workload"] == "prefill_fold_norm_fp8"
    rows = line["config"]["T"]
    assert line["value"] == pytest.approx(rows / (line["ms_per_step"] * 1e-3), rel=2e-3)
    rf = line["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s"
    assert rf["algorithmic_bytes_per_launch"] == 109_076_480
    assert rf["achieved"] == pytest.approx(
        rf["algorithmic_bytes_per_launch"] / (line["ms_per_step"] * 1e-3) / 1e9, rel=2e-3)
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"], rel=2e-3)
    assert 0.3 < rf["frac"] < 1.2
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0
    e2e = line["e2e"]
    assert e2e["unit"] == "tokens/s" and e2e["value"] > 0
    assert e2e["h2d_bytes_per_step"] == 4 * 2048 * 4096 * 2 + 2048 * 4096 * 2 + 4096 * 4
    assert e2e["d2h_bytes_per_step"] == 2048 * 4096 * 2 + 2048 * 4096 + 2048 * 4
    assert e2e["value"] < line["value"]            # host copies cost time
    assert line["gpu_launches"] == 20
    assert set(line["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}
    cfgs = line["configs"]
    assert len(cfgs) == 6 and all(c["us"] > 0 for c in cfgs.values())
    assert cfgs["cfg3_prefill_fp8_K4_T2048"]["us"] == pytest.approx(line["ms_per_step"] * 1e3,
                                                                    rel=2e-3)
