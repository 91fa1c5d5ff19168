"""bench.py's host-side logic, without a GPU: the source hash that keys the
recorded ncu traffic, the traffic lookup, the FLOP counts of the oracle
samples, the peaks file, and the parsing of the clock samples."""

import json
import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from exact_tiled_attention_08_gb300.workloads import WORKLOADS  # noqa: E402


def test_code_only_ignores_comments_and_whitespace():
    a = "int x = 1;  // one\n/* a block\n   comment */ int y=2;\n"
    b = "int x = 1;\n\n   int y=2;  // another comment"
    assert bench._code_only(a) == bench._code_only(b) == "int x = 1; int y=2;"
    assert bench._code_only("int x = 2;") != bench._code_only("int x = 1;")


@pytest.fixture
def fake_root(tmp_path, monkeypatch):
    src = os.path.join(ROOT, "exact_tiled_attention_08_gb300", "csrc")
    dst = tmp_path / "exact_tiled_attention_08_gb300" / "csrc"
    shutil.copytree(src, dst, ignore=shutil.ignore_patterns("*.o", "*.so"))
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "profiles" / "traffic.json"))
    return dst


def test_source_hash_follows_code_not_comments(fake_root):
    h_bwd, h_fwd = bench.kernel_source_hash("fa_bwd_kernel"), bench.kernel_source_hash("fa_fwd_kernel")
    with open(fake_root / "fa_bwd.cuh", "a") as f:
        f.write("\n// a new comment\n/* and another */\n")
    assert bench.kernel_source_hash("fa_bwd_kernel") == h_bwd
    with open(fake_root / "fa_bwd.cuh", "a") as f:
        f.write("\nnamespace fa { constexpr int kNewConstant = 1; }\n")
    assert bench.kernel_source_hash("fa_bwd_kernel") != h_bwd
    assert bench.kernel_source_hash("fa_fwd_kernel") == h_fwd  # fa_bwd.cuh is not a forward source
    # the host code is a source of every kernel
    with open(fake_root / "fa_lib.cu", "a") as f:
        f.write("\nstatic int g_unused_counter = 0;\n")
    assert bench.kernel_source_hash("fa_fwd_kernel") != h_fwd


def test_recorded_traffic_only_for_the_sources_it_was_taken_on(fake_root):
    entry = {"dram_bytes_per_launch": 123, "read": 100, "write": 23}
    d = {"fa_bwd_kernel": {"wl": dict(entry, source_hash=bench.kernel_source_hash("fa_bwd_kernel"))},
         "fa_fwd_kernel": {"wl": dict(entry, source_hash="0000000000000000")}}
    with open(bench.TRAFFIC_FILE, "w") as f:
        json.dump(d, f)
    assert bench.recorded_traffic("fa_bwd_kernel", "wl") == 123
    assert bench.recorded_traffic("fa_bwd_kernel", "other workload") is None
    assert bench.recorded_traffic("fa_fwd_kernel", "wl") is None  # stale hash
    with open(fake_root / "fa_bwd.cuh", "a") as f:
        f.write("\nnamespace fa { constexpr int kChanged = 2; }\n")
    assert bench.recorded_traffic("fa_bwd_kernel", "wl") is None  # the kernel changed since
    os.remove(bench.TRAFFIC_FILE)
    assert bench.recorded_traffic("fa_bwd_kernel", "wl") is None


def test_committed_traffic_file_is_well_formed():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    for kernel, per_wl in d.items():
        if kernel.startswith("_"):
            continue
        assert kernel in bench.KERNEL_SOURCES
        for wl, e in per_wl.items():
            assert wl in WORKLOADS
            assert e["dram_bytes_per_launch"] == e["read"] + e["write"] > 0
            assert len(e["source_hash"]) == 16


def test_sample_flops_match_the_workload_counts():
    for w in WORKLOADS.values():
        whole = bench.sample_flops(w, w.N) * w.B * w.H
        assert whole == pytest.approx(w.fwd_flops() + w.bwd_flops(), rel=1e-12)
    w = WORKLOADS["b4_h16_n2048_d128"]
    assert bench.sample_flops(w, 100) == pytest.approx(3.5 * 4 * w.d * 100 * w.N)
    c = WORKLOADS["causal_b2_h32_n8192_d128"]
    assert bench.sample_flops(c, 100) == pytest.approx(3.5 * 4 * c.d * 100 * 101 / 2)


def test_peaks_measured_or_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, src = bench.load_peaks()
    assert src == "fallback" and peaks == bench.FALLBACK_PEAKS
    with open(tmp_path / "MEASURED_PEAKS.json", "w") as f:
        json.dump({"hbm_gbs": 6790, "bf16_tflops": 1929, "bf16_tflops_sustained": 1712.9, "other": 1}, f)
    peaks, src = bench.load_peaks()
    assert src == "measured" and peaks == {"hbm_gbs": 6790.0, "bf16_tflops": 1929.0, "bf16_tflops_sustained": 1712.9}


class _FakeSmi:
    def __init__(self, out):
        self.out = out

    def terminate(self):
        pass

    def communicate(self, timeout=None):
        return self.out, ""


def test_clock_samples_parsed_with_throttle_reasons():
    s = bench.ClockSampler(0)
    s.proc = _FakeSmi("0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active\n"
                      "0, 2040, 2070, 1350.0, 0x4, Not Active, Not Active, Not Active, Active\n"
                      "0, 2070, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active\n"
                      "garbage line\n")
    info = s.stop()
    assert info == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    s.proc = _FakeSmi("0, 1500, 2070, 800, 0x8, Active, Not Active, Active, Not Active\n")
    assert s.stop()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    s.proc = None
    assert s.stop()["samples"] == 0
