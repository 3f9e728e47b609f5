"""Host logic of bench.py that needs no GPU: the clock sampler summarises only the samples
taken inside the timed region."""
import os
import sys
import tempfile

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _row(sm, max_sm, reasons=()):
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    flags = ", ".join("Active" if n in reasons else "Not Active" for n in names)
    return f"{sm}, {max_sm}, 900.0, 0x0, {flags}\n"


def test_clock_sampler_keeps_the_timed_region_only():
    sys.path.insert(0, ROOT)
    import bench

    cs = bench.ClockSampler(0)
    cs.proc = object()  # stands for the running nvidia-smi: only the file is read
    cs.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
    # before the timed region: idle clocks and a thermal flag that must not be reported
    cs.file.write(_row(600, 2070, ("hw_thermal_slowdown",)) + _row(610, 2070))
    cs.file.flush()
    cs.mark()
    # inside: the first row after the mark may be cut at the offset and is dropped
    cs.file.write(_row(1000, 2070, ("hw_slowdown",)) + _row(2040, 2070, ("sw_power_cap",)) + _row(2060, 2070))
    cs.file.flush()
    got = cs.summary()
    assert got["samples"] == 2
    assert got["sm_mhz"] == 2050.0 and got["sm_max_mhz"] == 2070.0
    assert got["reasons"] == ["sw_power_cap"]
    assert got["window"] == "timed region only"
    assert not os.path.exists(cs.file.name)


def test_clock_sampler_without_nvidia_smi():
    sys.path.insert(0, ROOT)
    import bench

    cs = bench.ClockSampler(0)
    cs.mark()  # no sampler running: nothing to mark
    assert cs.summary()["reasons"] == ["nvidia-smi unavailable"]


class _FakeNvml:
    """Stands for NvmlQueries: returns a scripted sequence of (sm_mhz, power_w, reason mask)."""

    def __init__(self, rows):
        self.rows = list(rows)
        self.max_mhz = 2070.0

    def sample(self, with_power):
        if not self.rows:
            return (2070.0, None, 0)
        mhz, pw, mask = self.rows.pop(0)
        return mhz, (pw if with_power else None), mask


def test_fast_clock_sampler_summarises_the_marked_window():
    sys.path.insert(0, ROOT)
    import bench

    fs = bench.FastClockSampler(_FakeNvml([]), period_s=0.0)
    # samples taken before mark(), inside the window, and after stop()
    fs.samples = [(600.0, 100.0, 0x40), (2000.0, 900.0, 0x0), (2040.0, None, 0x4), (2060.0, None, 0x0),
                  (500.0, None, 0x8)]
    fs.lo, fs.hi = 1, 4
    got = fs.summary()
    assert got["samples"] == 3
    assert got["sm_mhz"] == 2040.0 and got["sm_mhz_min"] == 2000.0 and got["sm_max_mhz"] == 2070.0
    assert got["reasons"] == ["sw_power_cap"]  # the thermal flag before and the slowdown after are outside
    assert got["power_w_max"] == 900.0
    assert got["window"] == "timed region only"


def test_fast_clock_sampler_thread_collects_between_mark_and_stop():
    sys.path.insert(0, ROOT)
    import time

    import bench

    fake = _FakeNvml([(1900.0 + i, 500.0, 0) for i in range(100000)])
    with bench.FastClockSampler(fake, period_s=0.0005) as fs:
        time.sleep(0.01)
        fs.mark()
        time.sleep(0.02)
        fs.stop()
        time.sleep(0.01)
    got = fs.summary()
    assert got["samples"] >= 5
    assert got["samples"] == fs.hi - fs.lo
    assert got["reasons"] == []


def test_reason_bits_name_the_rejected_slowdowns():
    sys.path.insert(0, ROOT)
    import bench

    assert set(bench.NVML_REASON_BITS.values()) == {"sw_power_cap", "hw_slowdown", "sw_thermal_slowdown",
                                                    "hw_thermal_slowdown"}


def test_reference_and_gpu_lines_share_the_config():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.line_config(1) == bench.line_config(1)
    assert bench.line_config(2)["parallelism"] == "replicas x2"
    assert bench.line_config(1)["seed"] == bench.SEED
