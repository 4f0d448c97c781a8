"""The bench's clock record on CPU: ClockSampler.summary over synthetic
nvidia-smi samples (the fields of its query, in order)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402

IDLE = ["Not Active"] * 4


def sample(sm, smax, watts, hw=False, hw_thermal=False, sw_thermal=False, power_cap=False):
    flags = ["Active" if f else "Not Active" for f in (hw, hw_thermal, sw_thermal, power_cap)]
    return [str(sm), str(smax), str(watts), "0x0000000000000000", *flags]


def sampler_with(samples):
    s = bench.ClockSampler(0)
    s.samples = list(samples)
    return s


def test_median_clock_and_max_inside_the_timed_region():
    rows = [(t, sample(mhz, 2070, w)) for t, mhz, w in
            ((10.0, 1000, 100), (11.0, 2070, 700), (11.5, 2060, 720), (12.0, 2070, 690),
             (13.5, 900, 90))]
    out = sampler_with(rows).summary(10.5, 12.5)
    assert out["source"] == "timed_region"
    assert out["samples"] == 3
    assert out["sm_mhz"] == 2070.0
    assert out["sm_max_mhz"] == 2070.0
    assert out["power_w_max"] == 720.0
    assert out["reasons"] == []


def test_throttle_reasons_are_reported_by_name():
    rows = [(1.0, sample(2070, 2070, 700)),
            (1.1, sample(1800, 2070, 1400, power_cap=True)),
            (1.2, sample(1500, 2070, 1390, hw_thermal=True, power_cap=True)),
            (1.3, sample(2070, 2070, 700, sw_thermal=True))]
    out = sampler_with(rows).summary(0.9, 1.4)
    assert out["reasons"] == ["hw_thermal_slowdown", "sw_power_cap", "sw_thermal_slowdown"]
    assert out["sm_mhz"] == (1800 + 2070) / 2


def test_short_region_widens_by_a_second():
    rows = [(4.2, sample(2070, 2070, 700)), (5.05, sample(2060, 2070, 710)),
            (5.8, sample(2050, 2070, 705)), (9.0, sample(100, 2070, 50))]
    out = sampler_with(rows).summary(5.0, 5.1)
    assert out["source"] == "timed_region_pm_1s"
    assert out["samples"] == 3
    assert out["sm_mhz"] == 2060.0


def test_no_samples_is_reported_as_unavailable():
    out = sampler_with([]).summary(0.0, 1.0)
    assert out["source"] == "unavailable" and out["samples"] == 0
    assert out["sm_mhz"] is None and out["reasons"] == []


def test_unparsable_fields_are_skipped():
    rows = [(1.0, ["[N/A]", "2070", "[N/A]", "0x0", *IDLE]),
            (1.1, ["2070", "[N/A]", "650", "0x0", *IDLE]),
            (1.2, ["2065", "2070", "640", "0x0", *IDLE])]
    out = sampler_with(rows).summary(0.5, 1.5)
    assert out["sm_mhz"] == (2070 + 2065) / 2
    assert out["sm_max_mhz"] == 2070.0
    assert out["power_w_max"] == 650.0
