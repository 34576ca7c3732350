"""The bench line's clock summary (no GPU): only nvidia-smi samples time-stamped
inside the timed region count, throttle reasons are collected from them, and a
region without any sample falls back to the whole sampler run, saying so."""
import datetime

import bench


def _line(ts, sm, power_cap=False, thermal=False):
    act = lambda b: "Active" if b else "Not Active"
    return (f"{ts}, 0, {sm}, 2070, 1200.00, 0x0000000000000000, Not Active, {act(thermal)}, "
            f"Not Active, {act(power_cap)}")


def _sampler(lines, begin, end):
    c = bench.ClockSampler(0)
    c.lines = lines
    c.t_begin, c.t_end = begin, end
    return c


def test_only_samples_inside_the_region_count():
    t0 = datetime.datetime(2026, 1, 2, 3, 4, 5)
    lines = [
        _line("2026/01/02 03:04:04.900", 900, thermal=True),   # before the region
        _line("2026/01/02 03:04:05.100", 2070, power_cap=True),
        _line("2026/01/02 03:04:05.150", 2055),
        _line("2026/01/02 03:04:05.200", 2040),
        _line("2026/01/02 03:04:06.500", 800, thermal=True),    # after the region
    ]
    s = _sampler(lines, t0, t0 + datetime.timedelta(seconds=1)).summary()
    assert s["samples"] == 3 and s["window"] == "timed region"
    assert s["sm_mhz"] == 2055 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]


def test_region_without_samples_uses_the_whole_run():
    t0 = datetime.datetime(2026, 1, 2, 3, 4, 5)
    lines = [_line("2026/01/02 03:04:04.900", 2070), _line("2026/01/02 03:04:05.900", 2070)]
    s = _sampler(lines, t0, t0 + datetime.timedelta(milliseconds=20)).summary()
    assert s["samples"] == 2 and s["window"].startswith("whole sampler run")


def test_no_samples_at_all():
    s = _sampler([], None, None).summary()
    assert s["samples"] == 0 and s["sm_mhz"] is None and s["reasons"] == []
