"""bench.py's clock record, on the CPU: the NVML summary when it has samples
of the timed region, else nvidia-smi's; and the NVML sampler reports itself
unavailable (instead of failing) where NVML cannot be loaded."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


class FakeNvml:
    ok = True

    def __init__(self, samples, max_mhz=2070.0, period=0.0005):
        self.samples, self.max_mhz, self.period = samples, max_mhz, period

    summary = bench.NvmlClockSampler.summary
    REASONS = bench.NvmlClockSampler.REASONS


class FakeSmi:
    def summary(self, t0, t1):
        return {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 1}


def test_nvml_samples_inside_the_window_make_the_record():
    # (time, SM MHz, reason bits, watts); 0x4 = sw_power_cap, 0x40 = hw_thermal_slowdown
    s = [(0.5, 1500.0, 0x40, 100.0), (1.1, 2070.0, 0x0, 300.0), (1.2, 2000.0, 0x4, 350.0),
         (1.3, 2070.0, 0x1, 320.0), (2.5, 900.0, 0x8, 50.0)]
    rec = bench.clock_record(FakeNvml(s), FakeSmi(), 1.0, 2.0)
    assert rec["samples"] == 3
    assert rec["sm_mhz"] == 2070.0 and rec["sm_max_mhz"] == 2070.0
    assert rec["reasons"] == ["sw_power_cap"]  # 0x1 (idle) is not a slowdown reason
    assert rec["power_w_max"] == 350.0
    assert rec["nvidia_smi"]["samples"] == 1


def test_falls_back_to_nvidia_smi():
    assert bench.clock_record(FakeNvml([(5.0, 2070.0, 0, 1.0)]), FakeSmi(), 1.0, 2.0)["samples"] == 1
    assert bench.clock_record(None, FakeSmi(), 1.0, 2.0)["samples"] == 1
    assert bench.clock_record(None, None, 1.0, 2.0) is None


def test_sampler_without_nvml_is_not_ok():
    s = bench.NvmlClockSampler(0)
    s.stop()
    if not s.ok:
        assert s.samples == []
