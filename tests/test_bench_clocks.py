"""bench.py's clock record: the summary of the 1 ms NVML samples and the decoding of NVML's
clock-event (throttle) reason bits, with a fake NVML library; no GPU."""
import ctypes

import bench


def test_fast_samples_summary():
    c = bench.ClockSampler(0)

    class FakeNvml:
        max_mhz = 2070.0

    c.nvml = FakeNvml()
    c.fast = [(2070.0, []), (2055.0, ["sw_power_cap"]), (2070.0, []), (2070.0, [])]
    s = c.summary()
    assert s["sm_mhz"] == 2070.0
    assert s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    assert s["samples"] == 4 and s["source"].startswith("NVML")


def test_no_samples_fallback_summary():
    s = bench.ClockSampler(0).summary()   # nothing sampled (no GPU here)
    assert s["sm_mhz"] is None and s["samples"] == 0 and s["reasons"] == []


def test_nvml_reason_bits():
    class FakeLib:
        def nvmlDeviceGetClockInfo(self, h, which, out):
            assert which == bench._Nvml.SM
            out._obj.value = 1980
            return 0

    def reasons(h, out):
        out._obj.value = 0x8 | 0x4 | 0x1   # hw_slowdown, sw_power_cap and an idle bit
        return 0

    n = bench._Nvml.__new__(bench._Nvml)
    n.c, n.lib, n.h, n.reasons_fn = ctypes, FakeLib(), ctypes.c_void_p(), reasons
    mhz, rs = n.sample()
    assert mhz == 1980.0
    assert sorted(rs) == ["hw_slowdown", "sw_power_cap"]
    assert bench.BAD_REASONS & set(rs) == {"hw_slowdown"}
