"""The bench's clock record on the CPU: samples are kept only inside the timed region, the
reasons of those samples are reported, and a region with no sample reports none.  A fake
reader stands in for NVML (the real one is read-only and needs a GPU driver)."""
import time

import bench


class FakeReader:
    def __init__(self, mhz, reasons):
        self.mhz, self.reasons = mhz, reasons

    def sample(self):
        return self.mhz, 2070.0, set(self.reasons)


def test_samples_inside_the_timed_region_only():
    rows = [(1.0, 2070.0, 2070.0, set()), (2.0, 1500.0, 2070.0, {"sw_power_cap"}),
            (3.0, 1600.0, 2070.0, {"sw_power_cap"}), (4.0, 2070.0, 2070.0, {"hw_slowdown"})]
    out = bench.summarize_clocks(rows, 1.5, 3.5, 1, "test")
    assert out["samples"] == 2 and out["sm_mhz"] == 1550.0
    assert out["reasons"] == ["sw_power_cap"]  # the hw_slowdown sample lies outside the region
    assert out["samples_around"] == 4 and out["reasons_around"] == ["hw_slowdown", "sw_power_cap"]
    assert out["sm_max_mhz"] == 2070.0


def test_region_without_samples():
    rows = [(1.0, 2070.0, 2070.0, set())]
    out = bench.summarize_clocks(rows, 5.0, 5.001, 20, "test")
    assert out["samples"] == 0 and out["sm_mhz"] is None and out["reasons"] == []


def test_polling_thread_with_a_fake_reader():
    c = bench.Clocks(0, reader=FakeReader(1800.0, {"sw_power_cap"}))
    c.start()
    c.begin()
    time.sleep(0.05)
    c.end()
    out = c.stop()
    assert out["source"] == "nvml" and out["period_ms"] == 1
    assert out["samples"] >= 5  # a 50 ms region polled every millisecond
    assert out["sm_mhz"] == 1800.0 and out["reasons"] == ["sw_power_cap"]


def test_reason_bits_follow_nvml():
    bits = bench.NvmlClockReader.BITS
    assert bits[0x4] == "sw_power_cap" and bits[0x8] == "hw_slowdown"
    assert bits[0x20] == "sw_thermal_slowdown" and bits[0x40] == "hw_thermal_slowdown"
