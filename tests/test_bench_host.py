"""Host logic of bench.py, without a GPU: the clock record of a timed window,
the peak each kernel's roofline is held against, the traffic taken from a
committed ncu summary only while the kernel's sources are unchanged, and
the config both arms of the benchmark print."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from onnx_lstm_gru_gb300 import workloads  # noqa: E402


def sampler_with(samples, windows):
    s = bench.ClockSampler(uuid=None)
    s.samples = list(samples)
    s.windows = dict(windows)
    s.sm_max = 2070.0
    s.source = "test"
    s._thread = object()  # as if NVML were sampling
    return s


def test_clock_window_uses_samples_inside_the_timed_region():
    samples = [(0.1 * i, 2070.0 if 10 <= i < 20 else 1200.0, 0) for i in range(30)]
    s = sampler_with(samples, {"w": [1.0, 1.95]})
    rec = s.window("w")
    assert rec["scope"] == "timed region" and rec["samples"] == 10
    assert rec["sm_mhz"] == 2070.0 and rec["reasons"] == []


def test_clock_window_falls_back_to_the_whole_run_when_too_few_samples():
    samples = [(0.1 * i, 2070.0, 0) for i in range(30)]
    s = sampler_with(samples, {"w": [1.0, 1.15]})  # 2 samples inside
    rec = s.window("w")
    assert rec["scope"] == "whole run" and rec["samples"] == 30


def test_clock_window_names_the_event_reasons_seen():
    # 0x4 sw_power_cap, 0x40 hw_thermal_slowdown (NVML's clock-event bits)
    samples = [(0.1 * i, 1900.0, 0x4 if i == 3 else (0x40 if i == 5 else 0)) for i in range(10)]
    s = sampler_with(samples, {"w": [0.0, 1.0]})
    assert s.window("w")["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def test_clock_median_ignores_idle_samples():
    samples = [(0.1 * i, v, 0) for i, v in enumerate([300.0, 300.0, 2070.0, 2070.0, 2000.0])]
    s = sampler_with(samples, {"w": [0.0, 1.0]})
    rec = s.window("w")
    assert rec["sm_mhz"] == 2070.0 and rec["samples_under_load"] == 3


PEAKS = {"f32": (78.0, "fp32 src"), "f16": (1800.0, "f16 src"), "bf16": (1900.0, "bf16 src")}


@pytest.mark.parametrize("kind,dtype,want", [("tensor", "f16", "f16"), ("tensor_small", "bf16", "bf16"),
                                             ("proj_tc", "f16", "f16"), ("fast", "f32", "f32"),
                                             ("fast", "f16", "f32"), ("grid", "f32", "f32")])
def test_roofline_peak_follows_the_kernel_and_its_operand_type(kind, dtype, want):
    r = bench.kernel_roofline(kind, 2e12, 1000.0, PEAKS, "no_such_workload", dtype)
    assert r["peak"] == PEAKS[want][0] and r["peak_source"] == PEAKS[want][1]
    assert r["bound"] == ("tensor" if kind in ("tensor", "tensor_small", "proj_tc") else "alu")
    assert r["achieved"] == pytest.approx(2.0) and r["frac"] == pytest.approx(2.0 / PEAKS[want][0])
    assert r["traffic"] is None  # no summary for this workload


def test_traffic_only_while_the_sources_are_unchanged(tmp_path, monkeypatch):
    name, files = bench.KERNEL_SOURCES["fast"]
    h = bench.kernel_source_hash(files)
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / f"{name}_wl.md").write_text(f"x\ndram_bytes_per_launch: 12345\nsource_hash: {h}\n")
    (prof / f"{name}_old.md").write_text("x\ndram_bytes_per_launch: 999\nsource_hash: 0123456789abcdef\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the sources are hashed under ROOT too: point the hash at the real tree
    monkeypatch.setattr(bench, "kernel_source_hash", lambda f: h)
    assert bench.profiled_traffic(name, "wl", h) == 12345.0
    assert bench.profiled_traffic(name, "old", h) is None
    assert bench.profiled_traffic(name, "missing", h) is None


def test_committed_profiles_carry_current_hashes_for_the_headline_kernels():
    """The headline layer's step and projection summaries describe the
    current sources (else the bench line's traffic would be null)."""
    w = workloads.HEADLINE
    for kind in ("fast", "proj_simt"):
        name, files = bench.KERNEL_SOURCES[kind]
        assert bench.profiled_traffic(name, w, bench.kernel_source_hash(files)) is not None, kind


def test_both_arms_print_the_same_config():
    w = workloads.WORKLOADS[workloads.HEADLINE]
    a = bench.config_of(w.name, w.problem, 1)
    b = bench.config_of(w.name, w.problem, 1)
    assert a == b and a["workload"] == w.name and a["seq"] == 80 and a["hidden"] == 256
    assert set(a) >= {"workload", "cell", "direction", "seq", "batch", "input", "hidden", "layout", "tensor_dtype"}


def test_other_configurations_are_the_named_workloads():
    for name in bench.SUB_WORKLOADS:
        assert name in workloads.WORKLOADS
    assert workloads.HEADLINE not in bench.SUB_WORKLOADS
