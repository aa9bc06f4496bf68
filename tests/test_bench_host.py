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


def test_targets_summary_from_components():
    comps = {"skinny_splitk_M16": {"roofline_frac": 0.712, "stream": {"roofline_frac": 0.80}},
             "swiglu_small_M2048": {"roofline_frac": 0.65, "stream": {"roofline_frac": 0.72}},
             "swiglu_small_M128": {"roofline_frac": 0.3, "stream": {"roofline_frac": 0.4}}}
    t = bench.targets(0.93, comps)
    assert t["gemm_8192"] == {"iso": 0.93, "b2b": 0.93, "target": 0.7, "pass": True}
    assert t["skinny_M16"]["pass"] is True and t["skinny_M16"]["b2b"] == 0.8
    assert t["swiglu_small_M2048"]["pass"] is False
    assert "target" not in t["swiglu_small_M128"]
    assert "skinny_M32" not in t                     # not measured: left out


def test_profiled_traffic_needs_the_current_digest(tmp_path, monkeypatch):
    import json
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    csrc = tmp_path / "swiglu_mlp_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in ("tc_gemm.cuh", "ptx.cuh", "launch_impl.cuh", "api.cu"):
        (csrc / name).write_text(f"int {name.split('.')[0]} = 1; // comment\n")
    dig = bench.kernel_source_digest()
    (prof / "k.json").write_text(json.dumps({"kernel_source_digest": dig,
                                             "dram_bytes_per_launch": 123.0}))
    assert bench.profiled_traffic("k.json") == 123.0
    # a comment-only change keeps the digest; a code change drops the figure
    (csrc / "api.cu").write_text("int api = 1; // another comment\n")
    assert bench.profiled_traffic("k.json") == 123.0
    (csrc / "api.cu").write_text("int api = 2;\n")
    assert bench.profiled_traffic("k.json") is None
    assert bench.profiled_traffic("missing.json") is None
