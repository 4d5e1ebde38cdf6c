"""Host logic of the benchmark, on CPU: the metric arithmetic, the roofline guard's ceilings, the
clock-record summary, the comment-insensitive sources hash and the rule that a recorded DRAM
traffic figure is used only while it was taken on the current sources."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_weight_gbps_and_pass_time():
    # 11.89 GB in 2.335 ms; the pages' 15.8 GB pass at 5 TB/s takes 3.16 ms
    assert bench.weight_gbps(11.89e9, 2.335) == pytest.approx(5092.1, abs=0.1)
    assert bench.ms_per_pass(5000.0) == pytest.approx(3.16)
    assert bench.weight_gbps(1e9, 1.0) == pytest.approx(1000.0)


def test_roofline_guard_ceilings(monkeypatch):
    g = bench.RooflineGuard()
    # no probe, no measured peak: the nominal spec
    monkeypatch.setattr(bench, "measured_peaks", lambda: None)
    assert g.ceiling() == bench.SPEC_HBM_GBS
    # the measured copy bandwidth plus 15 % (a read-only stream can beat a copy)
    monkeypatch.setattr(bench, "measured_peaks", lambda: {"hbm_gbs": 6775.9})
    assert g.ceiling() == pytest.approx(1.15 * 6775.9)
    # this run's read probe plus 3 % takes precedence
    g.read_gbps = 7000.0
    assert g.ceiling() == pytest.approx(7210.0)
    assert g.check(7200.0, "below") == 7200.0
    with pytest.raises(SystemExit, match="roofline guard"):
        g.check(7300.0, "above")


def test_clock_summary_names_every_reason_seen():
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.ok = True
    s.max_mhz = 2070
    s.samples = [(2070, 0), (2055, 0x4), (2070, 0x8), (1900, 0x4 | 0x40)]
    out = s.summary()
    assert out["sm_mhz"] == pytest.approx(2062.5)
    assert out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap"]
    assert out["samples"] == 4
    s.samples = []
    assert s.summary()["samples"] == 0


def _fake_tree(tmp_path, code):
    csrc = tmp_path / "bit_quantized_skinny_gb300" / "csrc"
    csrc.mkdir(parents=True, exist_ok=True)
    (csrc / "k.cu").write_text(code)
    return tmp_path


def test_sources_hash_ignores_comments_and_spacing(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(_fake_tree(tmp_path, "int f() { return 1; }\n")))
    h0 = bench.kernel_source_hash()
    _fake_tree(tmp_path, "// a comment\nint f()  {\n  return 1;   // another\n}\n")
    assert bench.kernel_source_hash() == h0
    _fake_tree(tmp_path, "int f() { return 2; }\n")
    assert bench.kernel_source_hash() != h0


def test_recorded_traffic_only_on_the_current_sources(monkeypatch, tmp_path):
    root = _fake_tree(tmp_path, "int f() { return 1; }\n")
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.recorded_traffic("q4k_tc_kernel", "pass64", 8) is None   # no record
    (root / "profiles").mkdir()
    rec = {"q4k_tc_kernel|pass64|M=8": {"dram_bytes_per_step": 123, "source_hash": bench.kernel_source_hash()}}
    (root / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("q4k_tc_kernel", "pass64", 8) == 123
    assert bench.recorded_traffic("q4k_tc_kernel", "pass64", 16) is None   # another workload
    _fake_tree(tmp_path, "int f() { return 2; }\n")                         # the kernel changed
    assert bench.recorded_traffic("q4k_tc_kernel", "pass64", 8) is None

