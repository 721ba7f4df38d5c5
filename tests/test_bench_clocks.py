"""bench.py's clock record: parsing of nvidia-smi samples and the timed-region window (CPU).

The timed region of the default run is well under a second, and the power cap can lower the
SM clock inside it for a few hundred milliseconds at a time, so the record keeps only the
samples taken inside the region and reports their median and minimum.
"""
import datetime
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

BASE = datetime.datetime(2026, 1, 1, 12, 0, 0)


def sampler_with(samples):
    """A ClockSampler holding the given (ms offset, sm MHz, power cap active) samples as
    nvidia-smi prints them (no process is started)."""
    c = bench.ClockSampler.__new__(bench.ClockSampler)
    c.t_start = c.t_end = None
    lines = []
    for ms, sm, cap in samples:
        t = (BASE + datetime.timedelta(milliseconds=ms)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        lines.append(f"{t}, {sm}, 2070, 812.25, 0x0000000000000004, Not Active, Not Active, "
                     f"Not Active, {'Active' if cap else 'Not Active'}")
    lines.append("garbage line")
    c.out = "\n".join(lines)
    return c


def at(ms):
    return BASE + datetime.timedelta(milliseconds=ms)


def test_only_samples_inside_the_timed_region_count():
    # idle at the max clock before and after, capped at 1740 MHz inside
    samples = [(50 * i, 1740 if 6 <= i <= 13 else 2070, 6 <= i <= 13) for i in range(20)]
    c = sampler_with(samples)
    c.t_start, c.t_end = at(290), at(660)
    s = c.summary()
    assert s["samples"] == 8
    assert s["sm_mhz"] == 1740 and s["sm_min_mhz"] == 1740 and s["sm_max_mhz"] == 2070
    assert s["frac_samples_below_max"] == 1.0
    assert s["reasons"] == ["sw_power_cap"]
    assert s["power_w_max"] == 812.25
    assert "inside the timed region" in s["sampling"]


def test_mixed_clocks_inside_the_region():
    samples = [(50 * i, 2070 if i % 2 else 1800, False) for i in range(10)]
    c = sampler_with(samples)
    c.t_start, c.t_end = at(0), at(450)
    s = c.summary()
    assert s["samples"] == 10
    assert s["sm_mhz"] == 1935.0 and s["sm_min_mhz"] == 1800
    assert s["frac_samples_below_max"] == 0.5
    assert s["reasons"] == []


def test_region_shorter_than_the_period_takes_the_nearest_sample():
    c = sampler_with([(0, 2070, False), (50, 1900, True), (100, 2070, False)])
    c.t_start, c.t_end = at(51), at(60)
    s = c.summary()
    assert s["samples"] == 1 and s["sm_mhz"] == 1900
    assert "nearest" in s["sampling"]


def test_unmarked_run_uses_every_sample_and_empty_output_is_unsampled():
    c = sampler_with([(0, 2070, False), (50, 1700, True)])
    assert c.summary()["samples"] == 2
    c.out = ""
    assert c.summary()["reasons"] == ["unsampled"]
