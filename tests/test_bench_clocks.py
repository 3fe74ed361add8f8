"""The benchmark's clock record on CPU: the NVML sampler's summary with a fake NVML device,
and the nvidia-smi fallback's CSV parsing.  Reading clocks is all either does; neither sets
anything on the GPU."""
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


class FakeNvml:
    """Stands in for bench._Nvml: a scripted sequence of (SM MHz, reasons) samples."""

    def __init__(self, samples, max_mhz=2070.0):
        self.samples = list(samples)
        self.max_mhz = max_mhz
        self.i = 0

    def sample(self):
        x = self.samples[min(self.i, len(self.samples) - 1)]
        self.i += 1
        return x


def test_nvml_summary_median_and_reasons():
    cs = bench.ClockSampler(0)
    cs.nvml = FakeNvml([(2070.0, set()), (1980.0, {"sw_power_cap"}), (2070.0, set())])
    with cs:
        time.sleep(0.05)
    out = cs.summary()
    assert out["samples"] >= 3
    assert out["sm_max_mhz"] == 2070.0
    assert out["sm_mhz"] == 2070.0                  # the median of mostly-max samples
    assert out["reasons"] == ["sw_power_cap"]
    assert out["source"].startswith("nvml")


def test_nvml_reason_bits():
    # the NVML clock-event bits the record reports, by name
    assert bench._Nvml.REASONS == {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                                   0x40: "hw_thermal_slowdown"}


def test_nvidia_smi_csv_parsing(tmp_path):
    cs = bench.ClockSampler(0)
    cs.nvml = None
    f = open(tmp_path / "clocks.csv", "w+")
    f.write("0, 2070 MHz, 2070 MHz, 900.1 W, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n")
    f.write("0, 1900 MHz, 2070 MHz, 1390.0 W, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n")
    f.write("0, 2070 MHz, 2070 MHz, 1000.0 W, 0x0000000000000040, Not Active, Active, Not Active, Not Active\n")
    f.write("garbage line\n")
    cs.out = f
    out = cs.summary()
    assert out["samples"] == 3
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert out["source"].startswith("nvidia-smi")


def test_no_gpu_gives_no_record():
    cs = bench.ClockSampler(0)
    cs.nvml = None
    with cs:
        pass
    # without nvidia-smi output there is no record rather than a made-up one
    out = cs.summary()
    assert out is None or out["samples"] >= 1
