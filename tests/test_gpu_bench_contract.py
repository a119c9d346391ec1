"""bench.py's JSON line on the GPU: one line per run with every key the benchmark contract names
(metric, value, the timing, roofline with its denominators, the oracle's CPU baseline, the
end-to-end figure with its copied bytes, the launch count and the clock record)."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-3000:]
    return json.loads(lines[0])


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


@pytest.mark.parametrize("config,dtype,flops", [("c3", "bf16", 2 * 8192 ** 3), ("c5", "nvfp4", 2 * 8192 ** 3)])
def test_bench_line_has_the_contract_keys(config, dtype, flops):
    steps = 8
    d = run_bench("--config", config, "--steps", str(steps), "--warmup", "3", "--e2e-steps", "3", "--cpu-seconds", "1")
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == 3 and d["dtype"] == dtype
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert abs(d["value"] - flops / (d["ms_per_step"] * 1e-3) / 1e12) < 1e-6 * d["value"]
    assert d["config"]["workload"].startswith(f"{dtype}_gemm_8192x8192x8192") and "l2_flush" in d["config"]
    assert "synthetic" in d["data"]
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9 and "traffic" in r
    assert r["instruction_rate"]["kernel_clock_mhz"] > 0
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["value"] > 0 and c["cores"] >= 1 and c["sample"] and c["unit"] == "TFLOP/s"
    e = d["e2e"]
    assert e["value"] > 0 and e["unit"] == "TFLOP/s" and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    launches_per_step = 2 if config == "c5" else 1  # row-major scales: the packing launch and the GEMM
    assert d["gpu_launches"] == steps * launches_per_step
    k = d["clocks"]["kernel"]
    assert k["launches_probed"] == steps and 300 < k["sm_mhz"] <= 2300
    assert "sm_max_mhz" in d["clocks"] and "reasons" in d["clocks"]
    assert d["vs_baseline"] is None or d["vs_baseline"] > 0
