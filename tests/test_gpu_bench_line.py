"""bench.py's GPU arm prints the one JSON line the benchmark contract asks
for: metric, unit and whole-job value, step timing, the roofline of the
dominant kernel against the measured copy peak, the end-to-end figure with
its host<->device bytes, clocks sampled during the timed region, the launch
count, and each op's own timing. A short run (3 timed steps) as a
subprocess, as the driver launches it."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OPS = ("compaction_fwd", "route_build", "binned_gather", "binned_scatter", "binned_wgrad", "padded_gather",
       "padded_scatter", "padded_wgrad", "compaction_bwd")


def test_bench_prints_the_contract_line():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3", "--warmup", "3",
                          "--no-cpu-baseline", "--e2e-steps", "2"], capture_output=True, text=True, timeout=900,
                         cwd=ROOT)
    assert res.returncode == 0, res.stderr[-3000:]
    lines = [ln for ln in res.stdout.strip().splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout[-2000:]
    d = json.loads(lines[0])
    sys.path.insert(0, ROOT)
    import bench

    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT and d["value"] > 0
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] == 3 and d["ms_per_step"] > 0
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["dtype"] == "bf16" and d["data"] == "synthetic"
    assert d["config"]["tokens"] == 8192 and "deepseek-v3" in d["config"]["workload"]
    # whole-job value = routed assignments per second of the timed steps
    assert abs(d["value"] - d["assignments_per_step"] / (d["ms_per_step"] * 1e-3)) <= 1e-3 * d["value"]
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0 and rf["kernel"] in d["kernels"]
    assert 0 < rf["frac"] < 1.2 and abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-3
    assert rf["traffic"] is None or rf["traffic"] > 0
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert e2e["value"] < d["value"]  # the host copies are inside its timed region
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    assert d["gpu_launches"] == 10 * d["steps"]
    for op in OPS:
        assert d["kernels"][op]["ms"] > 0
        assert d["kernels_alone"][op]["ms_median"] > 0
