"""Host-side pieces of bench.py: the algorithmic byte model the roofline
divides by, and the peak lookup (no GPU needed)."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from deterministic_mamba2_ssd_gb300.inputs import WORKLOADS  # noqa: E402


def test_api_bytes_of_the_16k_workload():
    # x, dout bf16 (2 x 512 MiB), B, C bf16 (2 x 32 MiB), dt fp32 (16 MiB), saved states fp32 (1 GiB)
    # read; dx fp32 (1 GiB), dB, dC fp32 (2 x 64 MiB), ddt (16 MiB) written; A, D, dA, dD
    w = WORKLOADS["bf16_T16384"]
    b = bench.api_bytes(w, 2)
    assert b == 3456111616
    assert b / (w.batch * w.seqlen) == pytest.approx(210945.0, abs=1.0)


def test_api_bytes_scale_with_tokens():
    a = bench.api_bytes(WORKLOADS["bf16_T2048"], 2)
    b = bench.api_bytes(WORKLOADS["bf16_T4096"], 2)
    assert b - a == pytest.approx(a - 3 * 256 * 4 - 2 * 256 * 4, rel=1e-12)


def test_peaks_from_the_measured_file_or_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_peaks() == (6800.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6784.2}))
    assert bench.load_peaks() == (6784.2, "measured")


def test_algorithmic_flops_of_the_pages_workloads():
    # per (chunk, head): 2 Q^2 P x 2 + 2 Q N P x 4; per (chunk, group): 2 Q^2 N x 3
    w = WORKLOADS["bf16_T16384"]
    per_head = 2 * 128 * 128 * 64 * 2 + 2 * 128 * 128 * 64 * 4
    per_group = 2 * 128 * 128 * 128 * 3
    assert bench.algorithmic_flops(w) == 128 * (256 * per_head + 8 * per_group)
    assert bench.algorithmic_flops(w) / 1e9 == pytest.approx(425.2, abs=0.05)
    assert bench.algorithmic_flops(WORKLOADS["bf16_varlen_T32768"]) / 1e9 == pytest.approx(837.5, abs=0.05)


def test_nominal_roofline_takes_the_slower_bound():
    w = WORKLOADS["bf16_T16384"]
    r = bench.nominal_roofline(w, 2, 1.0, 1950.0)
    assert r["bound"] == "hbm" and r["t_hbm_us"] == pytest.approx(432.0, abs=0.1)
    assert r["t_tensor_us"] == pytest.approx(218.1, abs=0.1)
    assert r["frac"] == pytest.approx(0.432, abs=1e-3)
    v = bench.nominal_roofline(WORKLOADS["bf16_varlen_T32768"], 2, 1.0, 1950.0)
    assert v["bound"] == "tensor" and v["roofline_us"] == pytest.approx(429.5, abs=0.2)


def test_tensor_peak_from_the_measured_file_or_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_tensor_peak() == (1900.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"bf16_tflops": 1872.3}))
    assert bench.load_tensor_peak() == (1872.3, "measured")
