"""The benchmark's clock record and roofline denominator on the CPU: the
in-process NVML poller against a stand-in NVML library (read calls only), the
merge with the nvidia-smi samples, and the choice between the burst and the
sustained peak."""
import ctypes
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


class FakeNvml:
    """Answers the four read calls the poller makes; records every call name so
    the test can check that nothing but reads were made."""

    def __init__(self, mhz=1965, max_mhz=2070, mask=0x4):
        self.mhz, self.max_mhz, self.mask = mhz, max_mhz, mask
        self.calls = []

    def nvmlDeviceGetHandleByUUID(self, uuid, out):
        self.calls.append("handle")
        return 0

    def nvmlDeviceGetClockInfo(self, dev, kind, out):
        self.calls.append("clock")
        ctypes.cast(out, ctypes.POINTER(ctypes.c_uint))[0] = self.mhz
        return 0

    def nvmlDeviceGetMaxClockInfo(self, dev, kind, out):
        self.calls.append("max")
        ctypes.cast(out, ctypes.POINTER(ctypes.c_uint))[0] = self.max_mhz
        return 0

    def nvmlDeviceGetCurrentClocksEventReasons(self, dev, out):
        self.calls.append("reasons")
        ctypes.cast(out, ctypes.POINTER(ctypes.c_ulonglong))[0] = self.mask
        return 0


def test_reason_bits():
    assert bench.nvml_reason_names(0) == []
    assert bench.nvml_reason_names(0x4) == ["sw_power_cap"]
    assert bench.nvml_reason_names(0x8 | 0x40 | 0x1) == ["hw_slowdown", "hw_thermal_slowdown"]
    assert bench.nvml_reason_names(0x20) == ["sw_thermal_slowdown"]


def test_poller_samples_inside_the_timed_region_only():
    fake = FakeNvml()
    with bench.NvmlPoller("GPU-x", 0, period_s=0.001, lib=fake) as p:
        time.sleep(0.02)             # before the timed region: not counted
        p.mark(True)
        fake.mhz = 1900
        time.sleep(0.03)
        p.mark(False)
        fake.mhz = 1000              # after it: not counted
        time.sleep(0.01)
    s = p.summary()
    assert s["samples"] >= 2
    assert s["sm_mhz"] == 1900 and s["sm_mhz_min"] == 1900 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
    assert set(fake.calls) <= {"handle", "clock", "max", "reasons"}


def test_poller_without_nvml_reports_no_samples():
    class Broken:
        def nvmlDeviceGetHandleByUUID(self, uuid, out):
            return 1

        def nvmlDeviceGetHandleByIndex_v2(self, i, out):
            return 1
    with bench.NvmlPoller("GPU-x", 0, lib=Broken()) as p:
        p.mark(True)
        p.mark(False)
    s = p.summary()
    assert s["samples"] == 0 and "no NVML handle" in s["error"]


def test_clock_record_prefers_the_timed_region():
    smi = {"sm_mhz": 1800.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 16}
    poll = {"samples": 12, "sm_mhz": 1950.0, "sm_max_mhz": 2070.0, "reasons": [],
            "sm_mhz_min": 1900.0, "at_start_mhz": 1950.0, "at_end_mhz": 1950.0,
            "period_ms": 2.0}
    r = bench.clocks_record(smi, poll, 3.0)
    assert r["sm_mhz"] == 1950.0 and r["reasons"] == ["sw_power_cap"] and r["soak_s"] == 3.0
    r2 = bench.clocks_record(smi, {"samples": 0}, 3.0)
    assert r2["sm_mhz"] == 1800.0 and r2["timed_region"] == {"samples": 0}


def test_peak_choice():
    peaks = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "measured"}
    p, kind = bench.choose_peak(peaks, 0.04)
    assert p == 1900.0 and "burst" in kind
    p, kind = bench.choose_peak(peaks, 3.0)
    assert p == 1700.0 and "sustained" in kind
