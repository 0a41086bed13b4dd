"""bench.py on CPU: its clock sampler against a fake NVML (the polling thread,
the timed-region filter and the clock-event reason bits; read-only queries, no
GPU), and the code hash that keys its traffic record."""
import ctypes
import threading
import time


class FakeNvml:
    """Answers the three queries the sampler makes; the SM clock and the reason
    bits are whatever the test sets."""

    def __init__(self):
        self.mhz, self.max_mhz, self.bits = 2070, 2070, 0
        self.shutdown = False

    def nvmlDeviceGetClockInfo(self, handle, clock, out):
        out._obj.value = self.mhz
        return 0

    def nvmlDeviceGetMaxClockInfo(self, handle, clock, out):
        out._obj.value = self.max_mhz
        return 0

    def reasons(self, handle, out):
        out._obj.value = self.bits
        return 0

    def nvmlShutdown(self):
        self.shutdown = True
        return 0


def _sampler(monkeypatch, lib):
    import bench
    s = bench.ClockSampler(0)
    monkeypatch.setattr(s, "_nvml_open", lambda: (ctypes, lib, None, lib.reasons))
    return s


def test_samples_inside_the_timed_region_only(monkeypatch):
    lib = FakeNvml()
    s = _sampler(monkeypatch, lib)
    lib.mhz = 1200                      # before the region: an idle clock that must not count
    s.start()
    time.sleep(0.05)
    lib.mhz, lib.bits = 2070, 0x4       # sw_power_cap: kept and noted
    t0 = time.time()
    time.sleep(0.05)
    t1 = time.time()
    lib.mhz, lib.bits = 900, 0x8        # after the region: a slowdown that must not count
    time.sleep(0.05)
    out = s.stop(t0, t1)
    assert lib.shutdown
    assert out["samples"] >= 5
    assert out["sm_mhz"] == 2070 and out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"]
    assert "timed region" in out["source"]


def test_throttle_bits_are_named():
    import bench
    s = bench.ClockSampler(0)
    s.nvml = (ctypes, FakeNvml(), None, None)
    s.stopping, s.thread = threading.Event(), threading.Thread(target=lambda: None)
    s.thread.start()
    s.samples = [(1.0, 2070, 2070, 0x8 | 0x40), (1.1, 2000, 2070, 0x20), (1.2, 1990, 2070, 0x1)]
    out = s.stop(0.5, 1.5)
    assert out["samples"] == 3 and out["sm_mhz"] == 2000
    assert out["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]   # 0x1 (idle) is not one


def test_region_shorter_than_the_poll_period_takes_the_nearest_sample():
    import bench
    s = bench.ClockSampler(0)
    s.nvml = (ctypes, FakeNvml(), None, None)
    s.stopping, s.thread = threading.Event(), threading.Thread(target=lambda: None)
    s.thread.start()
    s.samples = [(1.0, 1500, 2070, 0), (2.0, 2070, 2070, 0)]
    out = s.stop(1.9, 1.95)
    assert out["samples"] == 1 and out["sm_mhz"] == 2070
    assert "nearest" in out["source"]


def test_window_summarises_a_span_and_keeps_polling(monkeypatch):
    """window(t0, t1) gives the samples of one span while the sampler runs on
    (the timed region, then the GEMMs timed alone after it, from one sampler)."""
    lib = FakeNvml()
    s = _sampler(monkeypatch, lib)
    s.start()
    lib.mhz = 2070
    t0 = time.time()
    time.sleep(0.04)
    t1 = time.time()
    region = s.window(t0, t1)
    assert not lib.shutdown and s.thread.is_alive()
    lib.mhz, lib.bits = 1700, 0x4
    t2 = time.time()
    time.sleep(0.04)
    t3 = time.time()
    later = s.stop(t2, t3)
    assert lib.shutdown
    assert region["sm_mhz"] == 2070 and region["reasons"] == []
    assert later["sm_mhz"] == 1700 and later["reasons"] == ["sw_power_cap"]
    assert region["samples"] >= 3 and later["samples"] >= 3


def test_traffic_record_hash_covers_code_not_comments():
    """The traffic record's hash follows the kernels' code: a comment or a blank
    line changes nothing, a changed statement changes the hash."""
    import bench
    a = "int f(int x) {\n  return x + 1;   // one more\n}\n"
    b = "/* the successor */\nint f(int x) {\n\n  return x + 1;\n}\n// end\n"
    c = "int f(int x) {\n  return x + 2;   // one more\n}\n"
    assert bench.kernel_code(a) == bench.kernel_code(b)
    assert bench.kernel_code(a) != bench.kernel_code(c)
