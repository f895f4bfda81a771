"""The benchmark's JSON line on a GPU: every key the driver reads, with values
that hold together (a short run: 3 timed steps after 3 warm-up steps)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, cwd=ROOT, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_contract_keys(line):
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert k in line, k
    assert line["n_gpus"] == 1 and line["steps"] == 3 and line["warmup"] == 3
    assert line["higher_is_better"] is True and line["scaling"] == "weak" and line["vs_baseline"] is None
    assert "workload" in line["config"]


def test_values_hold_together(line):
    # value = P x params x 4 B per step over the step time
    n_bytes = 8 * line["config"]["params_per_worker"] * 4
    assert abs(line["value"] - n_bytes / (line["ms_per_step"] * 1e-3) / 1e9) <= 0.01 * line["value"]
    rf = line["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in rf, k
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s"
    assert 0.3 < rf["frac"] < 1.2 and abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    assert rf["traffic"] is not None, "the committed ncu summary no longer matches the kernel's sources"
    # 13 launches a step: per fusion buffer a range reset, a ring fold, a THC launch with the NMSE sums and
    # the kernel adding its CTAs' sums; one launch combining the buffers' sums
    assert line["gpu_launches"] == 13 * 3
    e2e = line["e2e"]
    # every worker's flat gradient buffer (tensors padded to 16-byte starts) crosses the link each step
    assert e2e["value"] > 0 and n_bytes <= e2e["h2d_bytes_per_step"] <= 1.001 * n_bytes
    assert e2e["d2h_bytes_per_step"] >= 8
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1
    assert line["clocks"] is None or "sm_mhz" in line["clocks"]
