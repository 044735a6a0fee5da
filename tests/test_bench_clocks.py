"""Host logic of bench.py's clock record: only nvidia-smi samples read while
the timed region ran count toward the median SM clock and the throttle
reasons (no GPU, no nvidia-smi: the sampler's lines are set by hand)."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


def _row(mhz, thermal="Not Active"):
    # index, clocks.sm, clocks.max.sm, power.draw, reasons.active,
    # hw_slowdown, hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap
    return f"0, {mhz}, 2070, 900.0, 0x0, Not Active, {thermal}, Not Active, Not Active"


def test_samples_outside_the_timed_region_are_left_out():
    import bench
    c = bench.ClockSampler(0)
    c.lines = [(0.90, _row(1000)), (1.01, _row(2070)), (1.03, _row(2070)),
               (1.05, _row(2060)), (1.30, _row(600, "Active"))]
    c.t_start, c.t_stop = 1.00, 1.04
    s = c.summary()
    assert s["window"] == "timed region"
    assert s["samples"] == 3          # 1.01, 1.03 and 1.05 (one period of slack)
    assert s["sm_mhz"] == 2070.0
    assert s["reasons"] == []         # the throttled sample came after the region


def test_region_shorter_than_the_period_takes_the_next_sample():
    import bench
    c = bench.ClockSampler(0)
    c.lines = [(0.90, _row(1000)), (1.10, _row(2040)), (1.30, _row(2070))]
    c.t_start, c.t_stop = 1.00, 1.005
    s = c.summary()
    assert s["samples"] == 1 and s["sm_mhz"] == 2040.0
    assert s["window"].startswith("first sample after")


def test_throttle_inside_the_region_is_reported():
    import bench
    c = bench.ClockSampler(0)
    c.lines = [(1.01, _row(1500, "Active")), (1.02, _row(2070))]
    c.t_start, c.t_stop = 1.00, 1.03
    assert c.summary()["reasons"] == ["hw_thermal_slowdown"]


def test_no_sampler_output_is_marked_unsampled():
    import bench
    c = bench.ClockSampler(0)
    c.t_start, c.t_stop = 1.0, 2.0
    s = c.summary()
    assert s["samples"] == 0 and s["reasons"] == ["unsampled"]
