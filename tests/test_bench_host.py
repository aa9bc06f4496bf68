"""Host logic of bench.py that needs no GPU: the clock sampler keeps only the
nvidia-smi samples whose timestamps fall inside the timed window, and reports
the throttle reasons seen there."""
import datetime
import os
import subprocess
import sys
import tempfile

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _row(t, sm, power, cap="Not Active", hw="Not Active"):
    stamp = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    # timestamp, index, clocks.sm, clocks.max.sm, power.draw, reasons.active,
    # hw_slowdown, hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap
    return f"{stamp}, 0, {sm}, 2070, {power}, 0x0, {hw}, Not Active, Not Active, {cap}\n"


def _sampler_with(rows):
    s = bench.ClockSampler(0, interval_ms=1)
    fd, s.path = tempfile.mkstemp(suffix=".csv")
    os.close(fd)
    with open(s.path, "w") as f:
        f.writelines(rows)
    s.out = open(os.devnull, "w")
    s.proc = subprocess.Popen([sys.executable, "-c", "import time; time.sleep(30)"])
    return s


def test_only_samples_inside_the_window_count():
    t0 = 1_800_000_000.0
    rows = [_row(t0 - 0.5, 2070, 150.0),                    # before: idle
            _row(t0 + 0.01, 1980, 900.0),
            _row(t0 + 0.03, 1960, 1100.0, cap="Active"),
            _row(t0 + 0.05, 1990, 1000.0),
            _row(t0 + 0.5, 2070, 200.0, hw="Active")]       # after: ignored
    out = _sampler_with(rows).stop(t0, t0 + 0.06)
    assert out["samples"] == 3
    assert out["sm_mhz"] == 1980.0
    assert out["reasons"] == ["sw_power_cap"]
    assert out["power_w_max"] == 1100.0
    assert abs(out["window_s"] - 0.06) < 1e-9


def test_no_sample_inside_the_window_gives_none():
    t0 = 1_800_000_000.0
    rows = [_row(t0 - 1.0, 2070, 150.0), _row(t0 + 1.0, 2070, 150.0)]
    assert _sampler_with(rows).stop(t0, t0 + 0.05) is None
