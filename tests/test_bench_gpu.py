"""bench.py's own arm on the GPU, in a short run: one JSON line carrying every
key of the output contract (metric, throughput, timing, roofline of the
dominant kernel with its measured traffic, end-to-end throughput with the
bytes copied per step, kernel launches, clocks, CPU baseline) and the
sub-measurements (forward workloads, packed batch, deterministic backward,
FP8 forward, decoding step), each with its roofline."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

pytestmark = pytest.mark.gpu


def test_bench_short_run_contract():
    steps = 3
    proc = subprocess.run([sys.executable, "bench.py", "--steps", str(steps), "--warmup", "3", "--e2e-steps", "2",
                           "--cpu-seconds", "1"], cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert proc.returncode == 0, proc.stderr[-3000:]
    lines = [json.loads(x) for x in proc.stdout.splitlines() if x.strip().startswith("{")]
    assert len(lines) == 1
    d = lines[0]
    assert d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == 3
    assert d["scaling"] == "weak" and d["dtype"] == "bf16" and d["data"].startswith("synthetic")
    assert d["config"]["workload"] == bench.WORKLOAD
    assert d["value"] > 0 and d["ms_per_step"] > 0
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["achieved"] > 0 and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert r["traffic"] is None or r["traffic"] > 0
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == "TFLOP/s"
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    # forward, pre-pass, main backward, dQ conversion per call
    assert d["gpu_launches"] == 4 * steps * d["config"]["calls_per_step"]
    c = d["clocks"]
    assert "sm_mhz" in c and "sm_max_mhz" in c and isinstance(c["reasons"], list)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0
    # every sub-measurement the line carries has its own roofline
    from exact_io_aware_29_gb300 import synth
    fw = d["forward_workloads"]
    assert set(fw) == set(synth.FORWARD_SWEEP)
    subs = [x["roofline"] for x in fw.values()]
    subs += [d["varlen"]["fwd_roofline"], d["varlen"]["bwd_roofline"], d["deterministic"]["roofline"],
             d["decode"]["roofline"]]
    subs += [d["fp8_forward"][k]["roofline"] for k in d["fp8_forward"] if isinstance(d["fp8_forward"][k], dict)]
    for x in subs:
        assert x["achieved"] > 0 and x["peak"] > 0 and abs(x["frac"] - x["achieved"] / x["peak"]) < 1e-9
    assert d["deterministic"]["bitwise_repeatable"] is True
