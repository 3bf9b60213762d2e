"""The pins are strong enough: plausible mistakes planted in a copy of the
oracle's C source (on the CPU) must each fail at least one pin.

Each mutant is the oracle with one edit: a wrong GQA head mapping, a window
off by one, a swapped page index, a dropped scale or normalisation, K used as
V, a sign error in the merge weights, a log-sum-exp without its log term, a
split that forgets where the attended range starts.
"""
import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "ref_decode.c")

MUTANTS = {
    "gqa_head_mapping": ("const int g = h / G;", "const int g = h % ly->Hkv;"),
    "window_off_by_one": ("? L - ly->window : 0;", "? L - ly->window - 1 : 0;"),
    "page_row_swapped": ("(size_t)(t % ly->P);", "(size_t)(t / ly->P);"),
    "scale_dropped": ("s[t - lo] = ly->scale * acc;", "s[t - lo] = acc;"),
    "normalisation_dropped": ("for (int i = 0; i < d; ++i) o[i] /= l;", ""),
    "k_used_as_v": ("load_row(ly, 1, b, g, t, row)", "load_row(ly, 0, b, g, t, row)"),
    "fp8_scale_dropped": ("row[i] = e4m3_to_f64(pool8[base + i]) * s;", "row[i] = e4m3_to_f64(pool8[base + i]);"),
    "fp8_exponent_bias": ("ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)"),
    "fp8_subnormal": ("ldexp((double)m, -9)", "ldexp((double)m, -10)"),
    "fp8_v_scale_from_k": ("(use_v ? ly->v_scale : ly->k_scale)", "(ly->k_scale)"),
    "merge_weight_sign": ("exp(lse[k] - M)", "exp(M - lse[k])"),
    "lse_without_log": ("*lse = m + log(l);", "*lse = m;"),
    "split_ignores_range_start": ("long long plo = (long long)lo + (long long)k * chunk;",
                                  "long long plo = (long long)k * chunk;"),
}


def _battery():
    """Run the main pins; return the names of those that fail."""
    failed = []
    checks = {
        "sdpa_gqa_window": lambda: pins.test_matches_library_sdpa(8, 2, 5),
        "sdpa_d256": lambda: pins.test_matches_library_sdpa(256, 4, 17),
        "shared_kv": lambda: pins.test_page_sizes_and_shared_kv(16, True),
        "page_size_1": lambda: pins.test_page_sizes_and_shared_kv(1, False),
        "hand_examples": pins.test_hand_examples,
        "zero_query": pins.test_zero_query_gives_mean_of_values,
        "split_merge": lambda: pins.test_split_merge_equals_unsplit(3, 17, 29),
        "split_merge_global": lambda: pins.test_split_merge_equals_unsplit(7, 5, 0),
        "lse": pins.test_lse_matches_scores,
        "window_invariant": pins.test_window_mask_invariant,
        "e4m3_codes": pins.test_e4m3_decoder_matches_torch_for_every_code,
        "fp8_sdpa": lambda: pins.test_fp8_decode_matches_sdpa_on_dequantized_kv(False, 0),
        "fp8_sdpa_kvshared": lambda: pins.test_fp8_decode_matches_sdpa_on_dequantized_kv(True, 9),
    }
    for name, fn in checks.items():
        try:
            fn()
        except (AssertionError, oracle.OracleError):
            failed.append(name)
    return failed


def _load_variant(src_text, workdir, tag):
    path_c = os.path.join(workdir, f"{tag}.c")
    path_so = os.path.join(workdir, f"{tag}.so")
    with open(path_c, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC",
                    "-o", path_so, path_c, "-lm"], check=True)
    lib = ctypes.CDLL(path_so)
    ref = oracle._load()
    for fn in ("ref_decode_rows", "ref_decode_split", "ref_merge", "ref_max_threads", "ref_decode_rows_fp8",
               "ref_e4m3_to_f64"):
        getattr(lib, fn).argtypes = getattr(ref, fn).argtypes
        getattr(lib, fn).restype = getattr(ref, fn).restype
    return lib


def test_unmutated_oracle_passes_battery():
    assert _battery() == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    with open(SRC) as f:
        text = f.read()
    old, new = MUTANTS[name]
    assert text.count(old) == 1, f"mutation site for {name} not unique"
    with tempfile.TemporaryDirectory() as tmp:
        lib = _load_variant(text.replace(old, new), tmp, name)
        monkeypatch.setattr(oracle, "_lib", lib)
        failed = _battery()
    assert failed, f"mutant {name} passed every pin"
