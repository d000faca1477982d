"""CPU tests of the benchmark's clock record: the NVML reason-mask decoding
(against a fake NVML library, read-only calls only), the parsing of
``nvidia-smi --query-gpu`` lines, and the summary that goes into the bench
line (median SM clock under load, every throttle reason seen)."""
import ctypes

import bench

NA, A = "Not Active", "Active"


class _FakeNvml:
    """Stands in for libnvidia-ml: fills the caller's out-arguments."""

    def __init__(self, mhz, mask, fail=False):
        self.mhz, self.mask, self.fail = mhz, mask, fail

    def nvmlDeviceGetClockInfo(self, dev, kind, ref):
        assert kind == 1                                  # NVML_CLOCK_SM
        if self.fail:
            return 999
        ref._obj.value = self.mhz
        return 0

    def reasons(self, dev, ref):
        ref._obj.value = self.mask
        return 0


def _poller(fake, max_mhz=2070.0):
    p = object.__new__(bench._NvmlPoller)               # no NVML init
    p.ct, p.lib, p.dev, p.max_mhz, p.rows = ctypes, fake, None, max_mhz, []
    p.reasons_fn = fake.reasons
    return p


def test_reason_mask_decoding():
    # NVML's clock-event bits: SwPowerCap 0x4, HwSlowdown 0x8,
    # SwThermalSlowdown 0x20, HwThermalSlowdown 0x40 (GpuIdle 0x1 ignored)
    cases = [(0x0, [NA, NA, NA, NA]), (0x1, [NA, NA, NA, NA]), (0x4, [NA, NA, NA, A]),
             (0x8, [A, NA, NA, NA]), (0x20, [NA, NA, A, NA]), (0x40, [NA, A, NA, NA]),
             (0x6C, [A, A, A, A])]
    for mask, want in cases:
        p = _poller(_FakeNvml(1980, mask))
        p._sample()
        assert p.rows == [(1980.0, 2070.0, want)], hex(mask)


def test_failed_read_adds_no_sample():
    p = _poller(_FakeNvml(1980, 0, fail=True))
    p._sample()
    assert p.rows == []


def test_summary_merges_nvml_and_smi_rows():
    s = bench.ClockSampler("0")
    s.rows = [(2070.0, 2070.0, [NA, NA, NA, A]), (2000.0, 2070.0, [NA, NA, NA, NA])]
    s.out = ("1900, 2070, 612.5, 0x0000000000000008, Active, Not Active, Not Active, Not Active\n"
             "not a sample\n"
             "N/A, 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
    d = s.summary()
    assert d["samples"] == 3
    assert d["sm_mhz"] == 2000.0 and d["sm_max_mhz"] == 2070.0
    assert d["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert d["source"] == "nvml 2 ms"


def test_summary_from_smi_only_and_unsampled():
    s = bench.ClockSampler("0")
    s.rows = None
    s.out = "\n".join(f"{m}, 2070, 700, 0x0, Not Active, Not Active, Not Active, Not Active"
                      for m in (2070, 2055, 2070, 1995))
    d = s.summary()
    assert d["samples"] == 4 and d["sm_mhz"] == 2070.0 and d["reasons"] == []
    assert d["source"] == "nvidia-smi 200 ms"
    s.out = ""
    assert bench.ClockSampler.summary(s) == {"sm_mhz": None, "sm_max_mhz": None,
                                             "reasons": ["unsampled"], "samples": 0}
