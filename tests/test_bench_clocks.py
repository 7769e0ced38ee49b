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


def test_clock_pass_record():
    # 2000 launches of 0.6 ms (1.2 s) of the 8192^3 GEMM at a median 1900 MHz
    flops = 2.0 * 8192 ** 3
    clocks = {"sm_mhz": 1900.0, "sm_min_mhz": 1800.0, "sm_max_mhz": 2070.0,
              "power_w_median": 1200.0, "power_w_max": 1390.0, "samples": 60,
              "reasons": ["sw_power_cap"]}
    peaks = {"hbm_gbs": 6663.6, "bf16_tflops": 1941.1, "bf16_tflops_sustained": 1728.9}
    r = bench.clock_pass_record(clocks, 2000, 1200.0, flops, peaks, False, 0.0, 152)
    want = flops / 0.6e-3 / 1e12
    assert abs(r["value"] - want) < 1e-6 and r["unit"] == "TFLOP/s"
    assert abs(r["frac_of_sustained_peak"] - want / 1728.9) < 1e-12
    assert abs(r["frac_of_nominal"] - want / 2250.0) < 1e-12
    assert abs(r["cycles_per_launch"] - 0.6e-3 * 1.9e9) < 1e-3
    pipe = 152 * 8192 * 1.9e9 / 1e12
    assert abs(r["pipe_peak_at_clock_tflops"] - pipe) < 1e-9
    assert abs(r["frac_of_pipe_peak_at_clock"] - want / pipe) < 1e-12
    assert r["samples"] == 60 and r["reasons"] == ["sw_power_cap"]
    # the skinny shape is judged against copy bandwidth
    nbytes = 541.1e6
    m = bench.clock_pass_record(clocks, 100, 10.0, 1.0, peaks, True, nbytes, 152)
    assert m["unit"] == "GB/s" and abs(m["value"] - nbytes * 100 / 0.01 / 1e9) < 1e-6
    assert "frac_of_nominal" not in m and abs(m["frac_of_hbm_gbs"] - m["value"] / 6663.6) < 1e-12
    assert "frac_of_pipe_peak_at_clock" not in m
