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
