"""The clock record of bench.py on CPU, from a recorded nvidia-smi stream: the
samples inside the timed region give the median SM clock and the active
throttle reasons; a timed region shorter than the sampling period takes the
nearest samples within 100 ms and says so; none at all is reported as such."""
import datetime
import os
import tempfile

import bench


def _row(t, sm, power=900.0, hw=False, cap=False):
    ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    act = "Active" if hw else "Not Active"
    capped = "Active" if cap else "Not Active"
    return "%s, 0, %d, 2070, %.2f, 0x0, %s, Not Active, Not Active, %s\n" % (
        ts, sm, power, act, capped)


def _sampler(lines, t0, t1):
    fd, path = tempfile.mkstemp(suffix=".csv")
    with os.fdopen(fd, "w") as f:
        f.writelines(lines)
    s = bench.ClockSampler(0)
    s.path, s.t0, s.t1 = path, t0, t1
    return s


def test_samples_inside_the_timed_region():
    t = 1_800_000_000.0
    lines = [_row(t - 0.5, 1000), _row(t + 0.1, 2000), _row(t + 0.2, 1900, cap=True),
             _row(t + 0.3, 2070), _row(t + 2.0, 500)]
    c = _sampler(lines, t, t + 0.35).stop()
    assert c["samples"] == 3 and c["sm_mhz"] == 2000 and c["sm_min_mhz"] == 1900
    assert c["sm_max_mhz"] == 2070 and c["reasons"] == ["sw_power_cap"]
    assert c["window"] == "inside the timed region"


def test_short_region_takes_the_nearest_samples():
    t = 1_800_000_000.0
    lines = [_row(t - 0.03, 2040), _row(t + 0.025, 2055, hw=True), _row(t + 0.5, 800)]
    c = _sampler(lines, t, t + 0.002).stop()
    assert c["samples"] == 2 and c["sm_mhz"] == (2040 + 2055) / 2
    assert c["reasons"] == ["hw_slowdown"]
    assert c["window"].startswith("nearest samples within 100 ms")


def test_no_sample_near_the_region():
    t = 1_800_000_000.0
    c = _sampler([_row(t - 5.0, 2070)], t, t + 0.002).stop()
    assert c["samples"] == 0 and c["sm_mhz"] is None
