"""The benchmark's clock summary (CPU): only nvidia-smi samples taken inside
the timed region enter the median SM clock that picks the roofline's peak."""
import datetime
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _line(t, sm, mx=2032, reasons=()):
    ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    flags = ["Active" if r in reasons else "Not Active" for r in bench.REASONS]
    return ", ".join([ts, str(sm), str(mx), "900.00"] + flags)


def test_summary_keeps_the_timed_region_only():
    c = bench.ClockSampler(None)
    t0 = 1_800_000_000.0
    # idle before (2032 MHz), busy at 1800-1900 under the power cap, idle after
    c.lines = ([_line(t0 + 0.05 * i, 2032) for i in range(6)] +
               [_line(t0 + 0.3 + 0.05 * i, 1800 + 20 * i, reasons=("sw_power_cap",)) for i in range(6)] +
               [_line(t0 + 0.6 + 0.05 * i, 2032, reasons=("hw_slowdown",)) for i in range(6)])
    c.t_start, c.t_end = t0 + 0.29, t0 + 0.56
    s = c.summary()
    assert s["samples"] == 6 and s["window"] == "timed region"
    assert s["sm_mhz"] == 1850.0 and s["sm_max_mhz"] == 2032.0
    assert s["reasons"] == ["sw_power_cap"]  # the idle samples' reasons are not counted


def test_summary_falls_back_to_all_samples():
    c = bench.ClockSampler(None)
    t0 = 1_800_000_000.0
    c.lines = [_line(t0, 1900), _line(t0 + 0.2, 2000), "garbage", ""]
    c.t_start, c.t_end = t0 + 0.05, t0 + 0.1  # shorter than the sampling interval
    s = c.summary()
    assert s["samples"] == 2 and s["window"] == "whole sampling period" and s["sm_mhz"] == 1950.0
    assert bench.ClockSampler(None).summary()["samples"] == 0
