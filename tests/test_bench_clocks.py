"""bench.py's clock record: only samples inside a long enough timed region describe it."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _row(mhz, watts, cap="Not Active"):
    return f"2026/01/01 00:00:00.000, {mhz}, 2070, {watts}, Not Active, Not Active, Not Active, {cap}"


def _sampler(rows):
    s = bench.ClockSampler(None, start=False)
    s.rows = rows
    return s


def test_long_region_reports_its_own_samples():
    # idle samples before and after, a loaded region from t = 10 to t = 11
    rows = [(t * 0.1, _row(2070, 190)) for t in range(100)]
    rows += [(10.0 + t * 0.1, _row(1600, 1390, "Active")) for t in range(11)]
    rows += [(11.2 + t * 0.1, _row(2070, 200)) for t in range(10)]
    s = _sampler(rows)
    s.t0, s.t1 = 10.0, 11.0
    out = s.summary()
    assert out["sm_mhz"] == 1600 and out["samples"] == 11
    assert out["reasons"] == ["sw_power_cap"] and out["power_w_median"] == 1390


def test_short_region_claims_no_clock():
    # an 11 ms region: the sample that happens to fall in it shows the idle clock before it
    rows = [(t * 0.1, _row(2070, 190)) for t in range(200)]
    s = _sampler(rows)
    s.t0, s.t1 = 10.05, 10.061
    out = s.summary(after=(10.2, 11.2))
    assert out["sm_mhz"] is None and out["power_w_median"] is None
    assert "no clock is claimed" in out["note"]
    assert out["sm_max_mhz"] == 2070
    assert out["after_region"]["samples"] == 10 and "continuation" in out["after_region"]["what"]


def _probe(records):
    """A clock-probe buffer (as the kernels write it) from (start_ns, start_clk, end_ns, end_clk) per CTA."""
    import torch
    buf = torch.zeros(4 * 8, dtype=torch.int64)
    for b, r in enumerate(records):
        buf[4 * b:4 * b + 4] = torch.tensor(r, dtype=torch.int64)
    return buf


def test_clock_probe_arithmetic():
    """Each CTA's clock is its clock64 difference over its %globaltimer difference; the
    median over the CTAs that recorded, and the span from the first start to the last end."""
    import dense_tensor_core_persistent_gb300 as g
    # 3 CTAs over 100 us at 1500, 1600 and 1800 MHz; unwritten slots stay zero
    recs = [(1_000_000, 5_000, 1_100_000, 5_000 + 150_000),
            (1_002_000, 9_000, 1_102_000, 9_000 + 160_000),
            (1_001_000, 7_000, 1_101_000, 7_000 + 180_000)]
    r = g.clock_probe_mhz(_probe(recs))
    assert r["ctas"] == 3
    assert abs(r["sm_mhz"] - 1600) < 1e-9 and abs(r["sm_mhz_min"] - 1500) < 1e-9 and abs(r["sm_mhz_max"] - 1800) < 1e-9
    assert abs(r["span_us"] - 102.0) < 1e-9
    assert g.clock_probe_mhz(_probe([]))["ctas"] == 0


def test_bench_summarizes_probed_launches():
    import dense_tensor_core_persistent_gb300 as g
    # (a start time of 0 marks an unwritten record: %globaltimer is never 0 on a running GPU)
    launches = [_probe([(1 + t, 0, 100_001 + t, mhz * 100)]) for t, mhz in ((0, 1700), (1, 1800), (2, 1750))]
    out = bench.summarize_probes(g, launches)
    assert out["launches_probed"] == 3 and out["ctas_per_launch"] == 1
    assert abs(out["sm_mhz"] - 1750) < 1e-6 and abs(out["sm_mhz_min"] - 1700) < 1e-6
    assert bench.summarize_probes(g, [_probe([])]) is None
