"""The pins are strong enough: plausible mistakes planted in a copy of the
oracle's C sources (on the CPU) must each fail at least one pin.

Each decode mutant is the oracle with one edit: a wrong GQA head mapping, a
window off by one, a swapped page index, a dropped scale or normalisation, K
used as V, a sign error in the merge weights, a log-sum-exp without its log
term, a split that forgets where the attended range starts, FP8 decoding
mistakes. Each mutant of the step before decode: a sum instead of a mean in
the norm, a dropped eps, a RoPE sign or partner error, a wrong frequency
exponent, the length used as the position, a swapped slot row, k normalised
with q's weight.
"""
import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
import test_oracle_pins as pins
import test_oracle_multi_pins as multi
import test_oracle_prepare_pins as prep

DECODE_SRC = os.path.join(os.path.dirname(oracle.__file__), "ref_decode.c")
PREPARE_SRC = os.path.join(os.path.dirname(oracle.__file__), "ref_prepare.c")

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
    "multi_position_off_by_one": ("const int pos = seq_lens[b] - T + j;", "const int pos = seq_lens[b] - T + j - 1;"),
    "multi_window_from_length": ("const int lo = (window > 0 && hi > window) ? hi - window : 0;",
                                 "const int lo = (window > 0 && seq_lens[b] > window) ? seq_lens[b] - window : 0;"),
    "multi_q_row_ignores_token": ("q + (size_t)r * d, lo, hi,", "q + ((size_t)b * T * Hq + h) * d, lo, hi,"),
}


PREPARE_MUTANTS = {
    "norm_sum_not_mean": ("sqrt(ms / d + eps)", "sqrt(ms + eps)"),
    "norm_eps_dropped": ("sqrt(ms / d + eps)", "sqrt(ms / d)"),
    "rope_sign": ("y[i] = x1 * c - x2 * s;", "y[i] = x1 * c + x2 * s;"),
    "rope_partner": ("const double x1 = y[i], x2 = y[i + half];", "const double x1 = y[i], x2 = y[i + 1];"),
    "rope_frequency": ("pow(theta, -2.0 * i / rot)", "pow(theta, -1.0 * i / rot)"),
    "position_is_length": ("const int pos = seq_lens[b] - 1;", "const int pos = seq_lens[b];"),
    "slot_row_swapped": ("slot_row[b] = pos % P;", "slot_row[b] = pos / P;"),
    "k_norm_with_q_weight": ("rms_norm(k_in + ((size_t)b * Hkv + g) * d, k_w,",
                             "rms_norm(k_in + ((size_t)b * Hkv + g) * d, q_w,"),
}


def _prepare_battery():
    """Run the pins of the step before decode; return the names of those that fail."""
    failed = []
    checks = {
        "hand_examples": prep.test_hand_examples,
        "complex_full": lambda: prep.test_rotation_equals_complex_multiplication(8, 8, 100.0, [1, 2, 9]),
        "complex_partial": lambda: prep.test_rotation_equals_complex_multiplication(256, 64, 1e6, [77, 65536]),
        "relative_position": prep.test_rotated_dot_depends_only_on_distance,
        "unit_mean_square": prep.test_normalised_rows_have_unit_mean_square,
        "pass_through": prep.test_pass_through_dims_beyond_rot,
        "slot": lambda: prep.test_slot_holds_the_newest_position(False, 16, [1, 16, 17, 100]),
        "slot_kv_shared": lambda: prep.test_slot_holds_the_newest_position(True, 16, [33, 2]),
        "rope_table": prep.test_rope_table_matches_closed_form,
    }
    for name, fn in checks.items():
        try:
            fn()
        except (AssertionError, oracle.OracleError, IndexError):
            failed.append(name)
    return failed


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
        "multi_sdpa": lambda: multi.test_multi_matches_library_sdpa_with_causal_mask(8, 4, 5, 3, 2, False),
        "multi_sdpa_global": lambda: multi.test_multi_matches_library_sdpa_with_causal_mask(8, 2, 0, 4, 16, False),
        "multi_is_decode": lambda: multi.test_token_j_is_decode_at_its_own_length(7),
    }
    for name, fn in checks.items():
        try:
            fn()
        except (AssertionError, oracle.OracleError):
            failed.append(name)
    return failed


def _load_variant(mutated_src, src_text, workdir, tag):
    """Build the oracle library with `mutated_src` replaced by `src_text`."""
    paths = []
    for src in oracle.SOURCES:
        path = os.path.join(workdir, f"{tag}_{os.path.basename(src)}")
        with open(path, "w") as f:
            if src == mutated_src:
                f.write(src_text)
            else:
                with open(src) as g:
                    f.write(g.read())
        paths.append(path)
    path_so = os.path.join(workdir, f"{tag}.so")
    subprocess.run(["gcc", *oracle.CFLAGS, "-o", path_so, *paths, "-lm"], check=True)
    lib = ctypes.CDLL(path_so)
    ref = oracle._load()
    for fn in ("ref_decode_rows", "ref_decode_split", "ref_merge", "ref_max_threads", "ref_decode_rows_fp8",
               "ref_e4m3_to_f64", "ref_decode_multi"):
        getattr(lib, fn).argtypes = getattr(ref, fn).argtypes
        getattr(lib, fn).restype = getattr(ref, fn).restype
    oracle.set_prepare_signatures(lib)
    return lib


def test_unmutated_oracle_passes_battery():
    assert _battery() == []
    assert _prepare_battery() == []


def _mutate(src, old, new):
    with open(src) as f:
        text = f.read()
    assert text.count(old) == 1, f"mutation site {old!r} not unique"
    return text.replace(old, new)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    text = _mutate(DECODE_SRC, *MUTANTS[name])
    with tempfile.TemporaryDirectory() as tmp:
        lib = _load_variant(DECODE_SRC, text, tmp, name)
        monkeypatch.setattr(oracle, "_lib", lib)
        failed = _battery()
    assert failed, f"mutant {name} passed every pin"


@pytest.mark.parametrize("name", sorted(PREPARE_MUTANTS))
def test_prepare_mutant_is_caught(name, monkeypatch):
    text = _mutate(PREPARE_SRC, *PREPARE_MUTANTS[name])
    with tempfile.TemporaryDirectory() as tmp:
        lib = _load_variant(PREPARE_SRC, text, tmp, name)
        monkeypatch.setattr(oracle, "_lib", lib)
        failed = _prepare_battery()
    assert failed, f"mutant {name} passed every pin"
