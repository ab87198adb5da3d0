"""bench.py's clock record, on CPU: the nvidia-smi samples taken during the
timed region are reduced to the median SM clock, the maximum clock and the
throttle reasons that were active (a fake sampler process stands in for
nvidia-smi)."""
from __future__ import annotations

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


class _Proc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


class _Thread:
    def join(self, timeout=None):
        pass


def sampler_with(lines, t_start, t_stop):
    s = bench.ClockSampler(0)
    s.proc, s._reader = _Proc(), _Thread()
    s.lines = lines
    s.t_start, s.t_stop = t_start, t_stop
    return s


def row(mhz, active="0x0000000000000000", hw="Not Active", hwt="Not Active", swt="Not Active", cap="Not Active"):
    return f"0, {mhz}, 2070, 1200.5, {active}, {hw}, {hwt}, {swt}, {cap}"


def test_only_samples_inside_the_timed_region_count():
    lines = [(1.0, row(1200, cap="Active")), (2.0, row(1800)), (2.5, row(1900)), (3.0, row(2000)),
             (9.0, row(600, hw="Active"))]
    rec = sampler_with(lines, 1.5, 3.5).stop()
    assert rec["sm_mhz"] == 1900 and rec["sm_max_mhz"] == 2070
    assert rec["reasons"] == [] and rec["samples"] == 3 and rec["window"] == "timed region"


def test_active_throttle_reasons_are_reported():
    lines = [(2.0, row(1700, cap="Active")), (2.1, row(1650, swt="Active")), (2.2, row(1690)),
             (2.3, row(1710, hwt="Active"))]
    rec = sampler_with(lines, 1.0, 3.0).stop()
    assert rec["reasons"] == ["hw_thermal_slowdown", "sw_power_cap", "sw_thermal_slowdown"]
    assert rec["sm_mhz"] == 1695


def test_malformed_samples_are_skipped_and_an_empty_window_falls_back():
    lines = [(5.0, "0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active"),
             (5.1, "garbage"), (5.2, row(1500))]
    rec = sampler_with(lines, 1.0, 2.0).stop()  # no sample inside the window
    assert rec["samples"] == 1 and rec["sm_mhz"] == 1500 and rec["window"] == "warm-up and timed region"
    assert sampler_with([(1.0, "garbage")], 0.0, 2.0).stop() is None
