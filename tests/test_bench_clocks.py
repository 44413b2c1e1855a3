"""bench.py's clock record: only nvidia-smi samples taken inside the timed
region count, and throttle reasons are collected from those samples."""
import datetime

import bench


class _FakeProc:
    def __init__(self, text):
        self.text = text

    def terminate(self):
        pass

    def communicate(self, timeout=None):
        return self.text, ""


def _line(t, sm, power, reasons=("Not Active",) * 4):
    stamp = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return ", ".join([stamp, str(sm), "2070", str(power), *reasons])


def test_samples_outside_the_window_are_dropped():
    t0 = 1_800_000_000.0
    lines = [_line(t0 - 0.25, 2070, 200.0),                       # before: idle
             _line(t0 + 0.05, 1800, 1390.0, ("Not Active",) * 3 + ("Active",)),
             _line(t0 + 0.10, 1750, 1395.0),
             _line(t0 + 0.15, 1700, 1400.0),
             _line(t0 + 0.60, 2070, 250.0, ("Active",) + ("Not Active",) * 3)]  # after
    c = bench.ClockSampler(0)
    c.proc = _FakeProc("\n".join(lines) + "\n")
    c.window(t0, t0 + 0.2)
    rec = c.stop()
    assert rec["samples"] == 3
    assert rec["sm_mhz"] == 1750 and rec["sm_min_mhz"] == 1700
    assert rec["power_w"] == 1395.0
    assert rec["reasons"] == ["sw_power_cap"]  # the hw_slowdown sample came after the region


def test_short_region_takes_the_nearest_samples():
    t0 = 1_800_000_000.0
    c = bench.ClockSampler(0)
    c.proc = _FakeProc(_line(t0 + 0.08, 1900, 1300.0) + "\n")
    c.window(t0, t0 + 0.01)
    assert c.stop()["samples"] == 1
