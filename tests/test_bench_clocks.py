"""bench.py's clock record keeps the nvidia-smi samples stamped inside the timed
region (a long prefill run can hit the power cap only while it is timed), and
falls back to every sample when the region is shorter than the 50 ms period or
the stamps cannot be read."""
import datetime
import os
import sys
import time

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _line(t, mhz, capped):
    ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    cap = "Active" if capped else "Not Active"
    return f"{ts}, {mhz}, 2070, 900.0, Not Active, Not Active, Not Active, {cap}"


def _sampler(now):
    c = bench.ClockSampler(0)
    c.lines = [_line(now - 0.3, 2070, False), _line(now - 0.2, 2070, False),
               _line(now, 1700, True), _line(now + 0.05, 1710, True),
               _line(now + 0.3, 2070, False)]
    return c


def test_samples_inside_the_timed_region_only():
    now = time.time()
    c = _sampler(now)
    c.t_start, c.t_stop = now - 0.01, now + 0.06
    s = c.summary()
    assert s["window"] == "timed region" and s["samples"] == 2
    assert s["sm_mhz"] == 1705.0 and s["reasons"] == ["sw_power_cap"]


def test_falls_back_to_every_sample():
    now = time.time()
    c = _sampler(now)
    s = c.summary()                                   # no region marked
    assert s["samples"] == 5 and s["window"] == "whole measurement"
    c.t_start, c.t_stop = now + 1.0, now + 1.01       # region between two samples
    s = c.summary()
    assert s["samples"] == 5 and s["window"].startswith("whole measurement")
    c.lines = [l.replace("/", "-", 2) for l in c.lines]   # unreadable stamps
    c.t_start, c.t_stop = now - 0.01, now + 0.06
    assert c.summary()["samples"] == 5


def test_clock_mark_sets_the_region_of_the_active_sampler_only():
    bench.clock_mark("start")                         # no active sampler: no effect
    c = bench.ClockSampler(0)
    bench._ACTIVE_SAMPLER = c
    try:
        bench.clock_mark("start")
        bench.clock_mark("stop")
    finally:
        bench._ACTIVE_SAMPLER = None
    assert c.t_start is not None and c.t_stop >= c.t_start
