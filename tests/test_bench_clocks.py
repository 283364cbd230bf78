"""Host logic of the benchmark's clock record: nvidia-smi samples are
timestamped and only those inside the timed region are summarised, so idle
samples before and after the region cannot hide a throttled clock."""
import datetime
import os
import sys
import time

sys.path.insert(0, os.path.join(os.path.dirname(__file__), ".."))
import bench  # noqa: E402


def sample_line(t, sm, watts, power_cap, thermal=False):
    ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    act = lambda b: "Active" if b else "Not Active"
    return (f"{ts}, 0, {sm}, 2070, {watts}, 0x4, Not Active, Not Active, {act(thermal)}, "
            f"{act(power_cap)}")


def fake_run(t0, n=40, load=range(12, 28), thermal_at=None):
    """Idle (2070 MHz, 150 W) except for the samples in `load` (1800 MHz, power capped)."""
    return "\n".join(sample_line(t0 + 0.05 * i, 1800 if i in load else 2070,
                                 1370 if i in load else 150, i in load, thermal=(i == thermal_at))
                     for i in range(n))


def test_window_keeps_only_the_timed_region():
    t0 = time.time()
    text = fake_run(t0)
    whole = bench.ClockSampler.summarize(text)
    assert whole["sm_mhz"] == 2070 and whole["samples"] == 40 and whole["window"] == "whole run"
    region = bench.ClockSampler.summarize(text, (t0 + 0.05 * 12 - 0.01, t0 + 0.05 * 27 + 0.01))
    assert region["window"] == "timed region"
    assert region["samples"] == 16 and region["sm_mhz"] == 1800 and region["power_w"] == 1370
    assert region["reasons"] == ["sw_power_cap"]


def test_short_region_takes_the_nearest_sample():
    t0 = time.time()
    text = fake_run(t0)
    s = bench.ClockSampler.summarize(text, (t0 + 0.05 * 20 + 0.01, t0 + 0.05 * 20 + 0.02))
    assert s["window"] == "nearest sample to the timed region"
    assert s["samples"] == 1 and s["sm_mhz"] == 1800


def test_throttle_reason_inside_the_region_is_reported():
    t0 = time.time()
    text = fake_run(t0, thermal_at=15)
    s = bench.ClockSampler.summarize(text, (t0 + 0.55, t0 + 1.4))
    assert "sw_thermal_slowdown" in s["reasons"]
    outside = bench.ClockSampler.summarize(text, (t0 + 0.9, t0 + 1.4))
    assert "sw_thermal_slowdown" not in outside["reasons"]


def test_malformed_lines_are_skipped():
    t0 = time.time()
    text = "garbage\n" + sample_line(t0, 1900, "[N/A]", False) + "\n, , ,\n"
    s = bench.ClockSampler.summarize(text)
    assert s["samples"] == 1 and s["sm_mhz"] == 1900 and "power_w" not in s
    assert bench.ClockSampler.summarize("") is None


def test_rejection_rule():
    ok = {"sm_mhz": 1800.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    assert not bench.clocks_rejected(ok)
    assert not bench.clocks_rejected(None)
    assert bench.clocks_rejected(dict(ok, reasons=["sw_power_cap", "hw_slowdown"]))
    assert bench.clocks_rejected(dict(ok, reasons=["sw_thermal_slowdown"]))
    locked = {"sm_mhz": 1200.0, "sm_max_mhz": 2070.0, "reasons": []}
    assert bench.clocks_rejected(locked)
    assert not bench.clocks_rejected(dict(locked, sm_mhz=2070.0))
