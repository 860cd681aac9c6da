"""bench.py's host-side rules on CPU: which FP8 peak the roofline divides by,
and that committed ncu figures are used only while the kernel sources they
were taken from are unchanged."""
import json
import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402

BURST, SUSTAINED = 3510.8, 2755.0


def test_short_region_takes_the_burst_peak():
    peak, rule = bench.choose_fp8_peak(140.0, {"sm_mhz": 1500.0, "sm_max_mhz": 2032.0}, BURST, SUSTAINED)
    assert peak == BURST and rule.startswith("burst")


def test_long_region_at_full_clock_takes_the_burst_peak():
    peak, rule = bench.choose_fp8_peak(5000.0, {"sm_mhz": 2000.0, "sm_max_mhz": 2032.0}, BURST, SUSTAINED)
    assert peak == BURST and "within 5%" in rule


def test_long_region_under_the_power_cap_takes_the_sustained_peak():
    peak, rule = bench.choose_fp8_peak(5000.0, {"sm_mhz": 1650.0, "sm_max_mhz": 2032.0}, BURST, SUSTAINED)
    assert peak == SUSTAINED and rule.startswith("sustained")


def test_long_region_without_clock_samples_takes_the_sustained_peak():
    peak, _ = bench.choose_fp8_peak(5000.0, {}, BURST, SUSTAINED)
    assert peak == SUSTAINED


def test_source_hash_covers_every_kernel_source(tmp_path, monkeypatch):
    """Editing any kernel source changes the hash that keys the ncu figures."""
    csrc = tmp_path / "fp8_fine_grained_20_b300" / "csrc"
    shutil.copytree(os.path.join(ROOT, "fp8_fine_grained_20_b300", "csrc"), csrc,
                    ignore=shutil.ignore_patterns("*.so", "__pycache__"))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    for name in ("ptx.cuh", "quant.cuh", "gemm.cuh", "gemm_mx.cuh", "swiglu.cuh", "fp8fg.cu"):
        p = csrc / name
        text = p.read_text()
        p.write_text(text + "\n// edit\n")
        assert bench.kernel_source_hash() != h0, name
        p.write_text(text)
    assert bench.kernel_source_hash() == h0


@pytest.mark.parametrize("matching", [True, False])
def test_ncu_figures_only_while_sources_unchanged(tmp_path, monkeypatch, matching):
    csrc = tmp_path / "fp8_fine_grained_20_b300" / "csrc"
    shutil.copytree(os.path.join(ROOT, "fp8_fine_grained_20_b300", "csrc"), csrc,
                    ignore=shutil.ignore_patterns("*.so", "__pycache__"))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "profiles").mkdir()
    record = {"source_hash": bench.kernel_source_hash() if matching else "0" * 16,
              "bytes_per_launch": {"grouped_gemm_moe": 2354400000},
              "tensor_pipe_active_pct": {"grouped_gemm_moe": 51.1}}
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps(record))
    if matching:
        assert bench.load_traffic() == {"grouped_gemm_moe": 2354400000}
        assert bench.load_tensor_pipe() == {"grouped_gemm_moe": 51.1}
    else:
        assert bench.load_traffic() == {}
        assert bench.load_tensor_pipe() == {}


def test_missing_ncu_record_gives_no_figures(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_traffic() == {}
    assert bench.load_tensor_pipe() == {}


def test_peaks_fall_back_when_the_measured_file_is_absent(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, source = bench.load_peaks()
    assert source == "fallback"
    assert set(peaks) >= {"hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"}


def test_measured_peaks_are_read(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"hbm_gbs": 6484.9, "bf16_tflops": 1755.4, "bf16_tflops_sustained": 1377.5}))
    peaks, source = bench.load_peaks()
    assert source == "measured"
    assert peaks == {"hbm_gbs": 6484.9, "bf16_tflops": 1755.4, "bf16_tflops_sustained": 1377.5}
