"""bench.py reads the measured HBM peak from a peaks record of several plausible
shapes, and falls back (and says so) when there is none (no GPU needed)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_flat_and_nested_records():
    assert bench.hbm_peak_from({"hbm_gbs": 7100.5, "bf16_tflops": 1900}) == 7100.5
    assert bench.hbm_peak_from({"hbm_GBs": 7000}) == 7000.0
    assert bench.hbm_peak_from({"hbm_copy_gbs": {"value": 6950.0}}) == 6950.0
    assert bench.hbm_peak_from({"gpu": "GB300", "peaks": {"hbm_gbs": 7050.0}}) == 7050.0
    assert bench.hbm_peak_from({"hbm": {"gbs": 6900.0}}) == 6900.0


def test_missing_or_malformed_records():
    assert bench.hbm_peak_from({"bf16_tflops": 1900}) is None
    assert bench.hbm_peak_from({"hbm_gbs": "n/a"}) is None
    assert bench.hbm_peak_from({"hbm_gbs": -1}) is None
    assert bench.hbm_peak_from([1, 2]) is None
    if not os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")):
        assert bench.measured_peaks() == (bench.FALLBACK_HBM_GBS, "fallback")
