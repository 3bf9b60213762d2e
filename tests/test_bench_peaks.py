"""bench.py's host logic, no GPU needed: it reads the measured HBM peak from a
peaks record of several plausible shapes and falls back (and says so) when
there is none; it rejects a timed region whose clock record shows a slowdown
or a clock lock."""
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


def test_clock_records_that_are_rejected():
    ok = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 5}
    assert not bench.clocks_rejected(ok)
    assert not bench.clocks_rejected(dict(ok, reasons=["sw_power_cap"], sm_mhz=1700.0))  # kept, noted
    assert bench.clocks_rejected(dict(ok, reasons=["hw_slowdown"]))
    assert bench.clocks_rejected(dict(ok, reasons=["sw_thermal_slowdown", "sw_power_cap"]))
    assert bench.clocks_rejected(dict(ok, sm_mhz=1500.0))  # well below max, no reason: a clock lock
    assert not bench.clocks_rejected({"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0})
