"""The benchmark's clock sampler (CPU, with a fake NVML): only samples taken inside the timed
region count, the median SM clock is reported, and throttle-reason bits map to their names."""

import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402


class FakeNvml:
    max_sm = 2070

    def __init__(self, script):
        self.script = list(script)

    def sample(self):
        return self.script.pop(0) if self.script else None


def _sampler(samples):
    cs = bench.ClockSampler.__new__(bench.ClockSampler)
    cs.rows, cs.window, cs._proc, cs._thread = [], None, None, None
    cs._nvml = FakeNvml([])
    cs.samples = samples
    return cs


def test_window_filters_samples():
    cs = _sampler([(0.0, 1200, 0x1), (1.0, 2070, 0), (1.5, 2040, 0x4), (2.0, 2070, 0), (9.0, 300, 0x1)])
    cs.mark(0.9, 2.1)
    got = cs.summary()
    assert got["samples"] == 3
    assert got["sm_mhz"] == 2070
    assert got["sm_max_mhz"] == 2070
    assert got["reasons"] == ["sw_power_cap"]


def test_thermal_and_slowdown_bits_are_named():
    cs = _sampler([(1.0, 1800, 0x8 | 0x40 | 0x80)])
    cs.mark(0.0, 2.0)
    assert cs.summary()["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_no_sample_inside_is_reported_unsampled():
    cs = _sampler([(5.0, 2070, 0)])
    cs.mark(0.0, 1.0)
    got = cs.summary()
    assert got["samples"] == 0 and got["reasons"] == ["unsampled"]
