"""The bench's clock sampling on the host: NVML reason bits, the summary object, and the
polling sampler against a stand-in reader (no GPU, no NVML)."""
import time

import bench


class FakeReader:
    def __init__(self, clocks, masks):
        self.clocks = list(clocks)
        self.masks = list(masks)
        self.i = 0

    def sm_mhz(self):
        v = self.clocks[min(self.i, len(self.clocks) - 1)]
        return v

    def sm_max_mhz(self):
        return 2070.0

    def reason_mask(self):
        m = self.masks[min(self.i, len(self.masks) - 1)]
        self.i += 1
        return m


def test_reason_bits():
    # nvml.h: SwPowerCap 0x4, HwSlowdown 0x8, SwThermalSlowdown 0x20, HwThermalSlowdown 0x40
    assert bench.reasons_from_mask(0) == []
    assert bench.reasons_from_mask(0x1) == []            # idle is not a slowdown
    assert bench.reasons_from_mask(0x4) == ["sw_power_cap"]
    assert bench.reasons_from_mask(0x8 | 0x40) == ["hw_slowdown", "hw_thermal_slowdown"]
    assert bench.reasons_from_mask(0x20) == ["sw_thermal_slowdown"]


def test_summary_median_and_union():
    s = bench.summarise_clocks([(2070.0, 2070.0, []), (1900.0, 2070.0, ["sw_power_cap"]),
                                (2000.0, 2070.0, [])])
    assert s == {"sm_mhz": 2000.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    assert bench.summarise_clocks([]) is None


def test_polling_sampler_collects_during_region():
    r = FakeReader([2070.0] * 3 + [1800.0] * 100, [0, 0, 0] + [0x4] * 100)
    sp = bench.PollingClockSampler(r, period=0.001)
    sp.start()
    time.sleep(0.05)
    out = sp.stop()
    assert out["samples"] >= 5 and out["source"] == "nvml"
    assert out["sm_max_mhz"] == 2070.0 and "sw_power_cap" in out["reasons"]


def test_polling_sampler_survives_reader_errors():
    class Broken(FakeReader):
        def sm_mhz(self):
            raise RuntimeError("query failed")
    sp = bench.PollingClockSampler(Broken([1.0], [0]), period=0.001)
    sp.start()
    time.sleep(0.01)
    assert sp.stop() is None
