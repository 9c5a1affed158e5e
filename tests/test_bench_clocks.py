"""The clock summary of bench.py: samples inside the timed region, or, for a
region shorter than the sampling period, the samples within 100 ms of it;
throttle reasons collected from the samples used."""
import datetime
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

ROWS = [
    "2026/12/03 10:00:00.000, GPU-a, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    "2026/12/03 10:00:00.050, GPU-a, 2040, 2070, 950.0, 0x4, Not Active, Not Active, Not Active, Active",
    "2026/12/03 10:00:00.050, GPU-b, 1000, 2070, 100.0, 0x0, Active, Not Active, Not Active, Not Active",
    "2026/12/03 10:00:00.400, GPU-a, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
]


def _sampler(tmp_path, t0_ms, t1_ms):
    c = bench.ClockSampler("GPU-a")
    c.proc = object()  # stands for the running nvidia-smi
    c.tmp = open(tmp_path / "clocks.csv", "w+")
    c.tmp.write("\n".join(ROWS) + "\n")
    base = datetime.datetime(2026, 12, 3, 10, 0, 0)
    c.t0 = base + datetime.timedelta(milliseconds=t0_ms)
    c.t1 = base + datetime.timedelta(milliseconds=t1_ms)
    return c


def test_samples_inside_the_timed_region(tmp_path):
    out = _sampler(tmp_path, 0, 60).summary()
    assert out["samples"] == 2 and "window" not in out
    assert out["sm_mhz"] == 2055.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]  # the other GPU's hw_slowdown is not ours


def test_short_region_takes_the_nearest_samples(tmp_path):
    out = _sampler(tmp_path, 60, 70).summary()
    assert out["samples"] == 2 and out["window"] == "within 100 ms of the timed region"
    assert out["reasons"] == ["sw_power_cap"]
