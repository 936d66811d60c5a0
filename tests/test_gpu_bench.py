"""The benchmark's GPU arm keeps its JSON contract: one line on rank 0 with
the headline value, the roofline of the dominant kernel, the CPU oracle
baseline, the end-to-end figure from host memory, the launch count and the
clocks seen during the timed region.  Run on the shrunken workload (the
256-token decode batch over a smaller pool) so it takes seconds."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu

STEPS, WARMUP = 5, 3


def _bench_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--small", "--no-detail",
                        "--steps", str(STEPS), "--warmup", str(WARMUP), "--cpu-seconds", "0.5"],
                       capture_output=True, text=True, cwd=ROOT, timeout=900)
    assert r.returncode == 0, r.stderr[-4000:]
    lines = [line for line in r.stdout.splitlines() if line.strip()]
    assert len(lines) == 1, r.stdout[-4000:]
    return json.loads(lines[0])


def test_gpu_arm_line():
    sys.path.insert(0, ROOT)
    import bench
    d = _bench_line()
    assert d["metric"] == bench.METRIC
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == STEPS and d["warmup"] == WARMUP
    assert d["scaling"] == "weak" and d["vs_baseline"] is None and d["data"] == "synthetic"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    # value: the batch's 256 new tokens over the mean step time (ms_per_step is
    # rounded to 10 ns)
    assert abs(d["value"] - 256 / (d["ms_per_step"] * 1e-3)) <= 2e-3 * d["value"]
    assert d["config"]["workload"] == bench.DECODE_DESC + " [small]"
    assert "flushed" in d["config"]["l2"]
    assert d["gpu_launches"] == STEPS * 3

    roof = d["roofline"]
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert roof["kernel"] in {"slot_mapping_paged_kernel", "slot_mapping_range_kernel",
                              "cache_write_kernel"}
    assert roof["achieved"] > 0 and roof["peak"] > 0
    # achieved = algorithmic bytes per launch / mean launch time (both printed
    # rounded: achieved to 0.1 GB/s, the time to 10 ns), frac = achieved / peak
    gbs = roof["alg_bytes_per_launch"] / (roof["avg_launch_us"] * 1e-6) / 1e9
    assert abs(roof["achieved"] - gbs) <= 0.05 + 2e-3 * gbs
    assert abs(roof["frac"] - gbs / roof["peak"]) <= 2e-3 * gbs / roof["peak"] + 1e-6
    peaks = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(peaks):
        assert roof["peak_kind"].startswith("measured")
    assert roof["traffic"] is None or roof["traffic"] > 0
    assert 0 < roof["frac_of_launch_floor"] <= 1.5

    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] == 1 and cpu["value"] > 0
    assert cpu["unit"] == "tokens/s" and cpu["sample"]

    e2e = d["e2e"]
    assert e2e["unit"] == "tokens/s" and e2e["value"] > 0
    assert e2e["h2d_bytes_per_step"] > 1 << 20  # the packed inputs, K/V rows included
    assert e2e["d2h_bytes_per_step"] >= 256 + 2 * 256 * 8  # error word and both slot maps

    clocks = d["clocks"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(clocks)
    assert isinstance(clocks["reasons"], list)

    pvr = d["paged_vs_range"]
    assert set(pvr["graph_replay_us"]) == {"paged", "range", "paged_fused", "range_fused"}
    assert d["gather_GBps"] > 0 and d["gather_roofline"]["frac"] > 0
    assert d["decode_step_with_gather"]["tokens_per_s"] > 0
