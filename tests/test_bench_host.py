"""Host logic of bench.py that decides how steps are timed (no GPU needed).

Timing rule: between timed steps either flush L2 or use inputs larger than
L2.  The headline flushes L2 before every step and takes the median of the
per-step times; block timing (K steps back to back between one pair of
events, no flush) is a side figure, allowed only when the step's inputs
exceed L2."""
import os
import sys
from types import SimpleNamespace

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

L2 = 136 * 10**6


@pytest.fixture(autouse=True)
def fake_l2(monkeypatch):
    monkeypatch.setattr(bench, "_l2_bytes", lambda dev: L2)


def _mode(timing, input_bytes):
    return bench._timing_mode(SimpleNamespace(timing=timing), input_bytes, None)


def test_headline_default_is_flushed():
    x_training_profile = 2 * 4096 * 20480          # 168 MB of BF16 X
    import sys as _s
    argv, _s.argv = _s.argv, ["bench.py"]
    try:
        args = bench._args()
    finally:
        _s.argv = argv
    assert args.timing == "flushed"
    assert _mode(args.timing, x_training_profile) == "flushed"
    assert args.steps >= 50                        # the median is over >= 50 flushed steps


def test_flushed_median_and_stats():
    import numpy as np
    times = [1.0, 3.0, 2.0, 100.0, 2.5]            # ms; one outlier
    st = bench._stats_us(times)
    assert st["reps"] == 5 and st["median_us"] == 2500.0
    assert st["min_us"] == 1000.0 and st["mean_us"] == np.mean(times) * 1e3


def test_explicit_modes():
    assert _mode("flushed", 10 * L2) == "flushed"
    assert _mode("block", L2 + 1) == "block"
    with pytest.raises(SystemExit):
        _mode("block", L2 // 2)                     # would time L2-resident inputs


def test_l2_note_names_the_rule_used():
    assert "not flushed" in bench._l2_note("block", 2 * L2, None)
    assert "flushed before every timed step" in bench._l2_note("flushed", 1, None)


# ------------------------------------------------------------------ clocks
def _sampler_with(lines):
    s = bench.ClockSampler(0)
    s.lines = list(lines)

    class _Done:   # stands for the finished nvidia-smi process
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    s.proc = _Done()
    return s


def test_clock_summary_median_max_and_reasons():
    # index, sm, max sm, power, active mask, hw, hw thermal, sw thermal, sw power cap
    lines = [
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1100.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    out = _sampler_with(lines).stop()
    assert out["samples"] == 3
    assert out["sm_mhz"] == 2070.0
    assert out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]


def test_clock_summary_flags_thermal_and_hw_slowdown():
    lines = ["0, 1500, 2070, 1400, 0x48, Active, Not Active, Active, Not Active"]
    out = _sampler_with(lines).stop()
    assert out["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert out["sm_mhz"] == 1500.0


def test_clock_summary_without_nvidia_smi():
    s = bench.ClockSampler(0)   # never started: no process
    out = s.stop()
    assert out["sm_mhz"] is None and out["reasons"] == ["nvidia-smi unavailable"]


# ------------------------------------------------------------------ ncu traffic, peaks, cores
def _fake_tree(tmp_path, traffic_hash):
    csrc = tmp_path / "rms_backward_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in bench._STREAMING_KERNEL_SOURCES:
        (csrc / name).write_text(f"// {name}\n")
    prof = tmp_path / "profiles"
    prof.mkdir()
    import json
    (prof / "ncu_traffic.json").write_text(json.dumps({
        "tcgen05": {"source_hash": traffic_hash, "dram_bytes_per_launch": 288057600}}))


def test_ncu_traffic_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _fake_tree(tmp_path, "0" * 16)
    assert bench._ncu_traffic("tcgen05") is None                 # stale capture
    current = bench._kernel_source_hash()
    import json
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps({
        "tcgen05": {"source_hash": current, "dram_bytes_per_launch": 288057600}}))
    assert bench._ncu_traffic("tcgen05") == 288057600.0
    assert bench._ncu_traffic("fma") is None                     # no capture for that kernel
    # any change to a streaming-kernel source makes the capture stale again
    (tmp_path / "rms_backward_gb300" / "csrc" / bench._STREAMING_KERNEL_SOURCES[0]).write_text("// edited\n")
    assert bench._ncu_traffic("tcgen05") is None


def test_peak_falls_back_without_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._peaks() == (bench.FALLBACK_HBM_GBS, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 6785.2}')
    assert bench._peaks() == (6785.2, "measured")


def test_cpu_clock_reports_cores_kept_busy():
    c = bench._CpuClock()
    assert c.cores() == 1.0          # nothing timed yet
    c.wall, c.cpu = 2.0, 28.0
    assert c.cores() == 14.0


def test_committed_traffic_capture_is_current():
    """profiles/ncu_traffic.json was taken on the streaming kernel's current
    sources, so the bench line carries its traffic figures; the SMs' L2
    writes equal the algorithmic dX + partial writes of the training profile."""
    import json
    assert bench._ncu_traffic("tcgen05") is not None
    d = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))["tcgen05"]
    T, K = 4096, 20480
    assert d["algorithmic_write_bytes"] == 2 * T * K + 8 * 24 * K * 4
    assert bench._ncu_l2_writes("tcgen05") == d["algorithmic_write_bytes"]


def test_cpu_worker_line(capsys):
    """The CPU-baseline child: one JSON line with per-run rates and cores."""
    import json
    assert bench._cpu_worker(json.dumps({"config": "tiny", "reps": 2, "seconds": 0.05})) == 0
    d = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert len(d["gbs"]) == 2 and all(v > 0 for v in d["gbs"])
    assert d["T_full"] == 64 and d["K"] == 512 and d["impl"]
