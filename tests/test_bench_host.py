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
