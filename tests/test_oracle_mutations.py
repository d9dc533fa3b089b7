"""Plant plausible mistakes in a scratch copy of the oracle and check the pins catch them.

Each mutation edits the C source text in a temporary directory, compiles it,
and points the oracle wrapper at the mutant; the committed oracle is untouched.
Every mutant must fail at least one of the pin tests, showing the pins are
strong enough to expose a dropped term, a wrong index or a misaligned mask.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
import tests.test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTATIONS = {
    "interleaved_gqa": ("int g = h / G;", "int g = h % J->Hkv;"),
    "scale_dropped": ("s[j] = scale * acc;", "s[j] = acc;"),
    "causal_off_by_one": ("int64_t visible = J->causal ? pos + 1 : n;", "int64_t visible = J->causal ? pos : n;"),
    "noncausal_flag_ignored": ("int64_t visible = J->causal ? pos + 1 : n;", "int64_t visible = pos + 1;"),
    "page_slot_shift": ("int64_t slot = j % J->ps;", "int64_t slot = (j + 1) % J->ps;"),
    "lse_without_max": ("*lse = m + log(l);", "*lse = log(l);"),
    "prefill_top_left_causal": ("visible = r + Lk - Lq + 1;", "visible = r + 1;"),
    "head_and_slot_strides_swapped": ("slot * J->ks[1] + (int64_t)g * J->ks[2]",
                                      "slot * J->ks[2] + (int64_t)g * J->ks[1]"),
    "missing_normalisation": ("for (int d = 0; d < dv; ++d) out[d] /= l;", ""),
    "fp8_value_scale_dropped": ("out[d] += p * (v_scale * oracle_e4m3_to_double", "out[d] += p * (oracle_e4m3_to_double"),
    "fp8_exponent_bias_off": ("else v = ldexp(1.0 + m / 8.0, e - 7);", "else v = ldexp(1.0 + m / 8.0, e - 8);"),
    "window_off_by_one": ("first = pos - J->window_left;", "first = pos + 1 - J->window_left;"),
    "append_clamp_after_base": ("if (slot < 0) slot = 0;                      /* clamp first ... */\n            int64_t row = layer_base + slot;",
                                "int64_t row = layer_base + slot;\n            if (row < 0) row = 0;"),
    "append_fp8_scale_multiplied": ("oracle_e4m3_from_float(x / sc)", "oracle_e4m3_from_float(x * sc)"),
}

PIN_CHECKS = [
    lambda: pins.test_decode_matches_sdpa_on_dense_copy(1, (5, 1, 13), 4, "random"),
    lambda: pins.test_decode_matches_sdpa_on_dense_copy(3, (7, 9, 12), 4, "random"),
    pins.test_prefill_matches_sdpa_per_sequence,
    pins.test_seq_len_one_returns_that_value_row,
    pins.test_two_key_closed_form,
    pins.test_gqa_mapping_worked_example,
    pins.test_lse_bounds,
    pins.test_e4m3_decoding_matches_torch_for_every_byte,
    lambda: pins.test_fp8_kv_decode_matches_sdpa_on_dequantized_copy(1, (5, 1, 13)),
    lambda: pins.test_window_matches_sdpa_on_dense_copy(2, (9, 30, 2), 4, 7),
    pins.test_window_zero_sees_own_position_only,
    lambda: pins.test_noncausal_decode_matches_masked_sdpa(-1),
    pins.test_warmup_slot_is_clamped_before_the_layer_base,
    lambda: pins.test_append_changes_only_the_addressed_rows(True),
]


def _compile_mutant(tmp_path, name):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / f"lib{name}.so"
    subprocess.check_call(["gcc", "-O1", "-fPIC", "-shared", "-pthread", "-o", str(lib), str(path), "-lm"])
    return str(lib)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutant(tmp_path, monkeypatch, name):
    lib_path = _compile_mutant(tmp_path, name)
    oracle._load()                                   # fetch argtypes from the real library
    real = oracle._lib
    mutant = ctypes.CDLL(lib_path)
    for fn in ("oracle_paged_decode", "oracle_paged_decode_kv8", "oracle_paged_decode_window",
               "oracle_paged_decode_masked", "oracle_e4m3_to_double", "oracle_varlen_prefill",
               "oracle_e4m3_from_float", "oracle_kv_append"):
        getattr(mutant, fn).restype = getattr(real, fn).restype
        getattr(mutant, fn).argtypes = getattr(real, fn).argtypes
    monkeypatch.setattr(oracle, "_lib", mutant)
    caught = 0
    for check in PIN_CHECKS:
        try:
            check()
        except (AssertionError, ValueError):
            caught += 1
    assert caught >= 1, f"no pin caught mutation {name}"
