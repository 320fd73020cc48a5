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
