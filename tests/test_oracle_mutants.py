"""The pins have teeth: each planted mistake in a copy of the oracle's C
source (a tie broken upward, a wrong emax or bias, swapped nibbles, a lost
sign, a dropped accumulator term, a reversed operand index ...) must make at
least one pin in test_oracle_pins.py fail.  The mistakes are planted on the
CPU, in a temporary copy; the real oracle source is never touched."""
import os
import shutil
import subprocess

import pytest

import oracle
from oracle import build as obuild
import test_oracle_next as nxt
import test_oracle_pins as pins

E2M1, E4M3 = oracle.E2M1, oracle.E4M3

MUTANTS = {
    "ties_go_up": ("if (d < best_d) {", "if (d <= best_d) {"),
    "emax_e2m1": ("return fmt == MXO_E2M1 ? 2 : 8;", "return fmt == MXO_E2M1 ? 3 : 8;"),
    "emax_e4m3": ("return fmt == MXO_E2M1 ? 2 : 8;", "return fmt == MXO_E2M1 ? 2 : 7;"),
    "nibbles_swapped": ("(uint8_t)((hi << 4) | lo)", "(uint8_t)((lo << 4) | hi)"),
    "e2m1_sign_bit": ("return fmt == MXO_E2M1 ? 0x8 : 0x80;", "return fmt == MXO_E2M1 ? 0x4 : 0x80;"),
    "scale_bias_store": ("*scale = (uint8_t)(e + 127);", "*scale = (uint8_t)(e + 128);"),
    "scale_bias_decode": ("return ldexp(1.0, byte - 127);", "return ldexp(1.0, byte - 126);"),
    "clip_low": ("if (e < -127) e = -127;", "if (e < -126) e = -126;"),
    "no_nan_scale": ("if (byte == 0xFF) return NAN;", "if (byte == 0x1FF) return NAN;"),
    "floor_log2_off": ("(void)frexp(v, &ex);\n    return ex - 1;", "(void)frexp(v, &ex);\n    return ex;"),
    "e4m3_subnormal": ("return ldexp((double)M, -9);", "return ldexp((double)M, -10);"),
    "zero_block_scale": ("*scale = 127;\n        return;", "*scale = 0;\n        return;"),
    "signed_amax": ("double a = fabs((double)x[i]);", "double a = (double)x[i];"),
    "gemm_drops_c0": ("double acc = c0, s = 0.0;", "double acc = 0.0, s = 0.0;"),
    "gemm_b_reversed": ("deq_exact(b_fmt, rb, sb, k);", "deq_exact(b_fmt, rb, sb, K - 1 - k);"),
    "sign_of_small_negatives": ("if (x[i] < 0.0f) code |= sign_bit_of(fmt);",
                                "if (x[i] < 0.0f && best) code |= sign_bit_of(fmt);"),
}

PIN_CALLS = [
    (pins.test_e2m1_decode_matches_page_table, {}),
    (pins.test_e2m1_decode_matches_bit_formula, {}),
    (pins.test_e4m3_decode_matches_torch_all_codes, {}),
    (pins.test_e8m0_decode_matches_torch_and_page, {}),
    (pins.test_floor_log2_matches_bit_extraction, {}),
    (pins.test_zero_block_gives_zero_codes_and_scale_127, {}),
    (pins.test_low_nibble_holds_element_zero, {}),
    (pins.test_tie_rule_lower_magnitude, {}),
    (pins.test_rounding_at_every_midpoint_against_exact_argmin, {"fmt": E2M1}),
    (pins.test_rounding_at_every_midpoint_against_exact_argmin, {"fmt": E4M3}),
    (pins.test_scale_clip_low_and_subnormal_codes, {}),
    (pins.test_negative_values_and_signed_zero, {}),
    (pins.test_nan_scale_poisons_whole_block, {}),
    (pins.test_gemm_integer_case_is_exact, {}),
    (pins.test_gemm_factored_block_sums, {"fa": E4M3, "fb": E2M1}),
    (pins.test_gemm_operand_orientation, {}),
]


# mistakes in the functions beyond the three core ops, against their own pins
MUTANTS_NEXT = {
    "axis0_gather_transposed": ("blockv[i] = x[(b * MXO_BLOCK + i) * cols + c];",
                                "blockv[i] = x[c * rows + b * MXO_BLOCK + i];"),
    "bf16_ties_away": ("if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) r = keep + 1u;",
                       "if (rest >= 0x8000u) r = keep + 1u;"),
    "bf16_truncates": ("if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) r = keep + 1u;",
                       "if (rest > 0xFFFFu) r = keep + 1u;"),
    "f32b_b_transposed": ("* (double)B[k * N + n];", "* (double)B[n * K + k];"),
    "f32b_drops_c0": ("double acc = (double)C0[m * N + n], s = 0.0;", "double acc = 0.0, s = 0.0;"),
    "fold_touches_nan": ("if (b == 0xFF) continue;", "if (b == 0x1FF) continue;"),
    "fold_saturates_at_255": ("if (b > 254) b = 254;", "if (b > 255) b = 255;"),
    "fold_wraps_low": ("if (b < 0) b = 0;", "if (b < 0) b += 256;"),
    "fold_exponent_off": ("return ex - 1;\n}\n\nint mxo_num_threads", "return ex;\n}\n\nint mxo_num_threads"),
}

PIN_CALLS_NEXT = [
    (nxt.test_axis0_is_quantize_of_the_transpose, {"fmt": E4M3, "rows": 64, "cols": 33}),
    (nxt.test_axis0_literal_column, {}),
    (nxt.test_dequantize_bf16_every_code_and_scale, {"fmt": E4M3}),
    (nxt.test_dequantize_bf16_literals, {}),
    (nxt.test_f32b_matches_numpy, {"fmt": E2M1, "M": 17, "N": 9, "K": 96}),
    (nxt.test_f32b_equals_mx_product_when_b_is_representable, {}),
    (nxt.test_fold_scale_multiplies_by_power_of_two, {"fmt": E4M3}),
    (nxt.test_fold_scale_saturates_and_keeps_nan, {}),
    (nxt.test_fold_exponent, {}),
]


@pytest.fixture(scope="module")
def src_text():
    with open(obuild.SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, src_text, tmp_path):
    old, new = MUTANTS[name]
    assert src_text.count(old) == 1, f"mutation anchor for {name} not unique"
    src = tmp_path / "mutant.c"
    src.write_text(src_text.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run([obuild._cc(), "-std=c99", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
                    str(src), "-o", str(lib), "-lm"], check=True)
    caught = []
    with oracle.use_library(str(lib)):
        for fn, kw in PIN_CALLS:
            try:
                fn(**kw)
            except (AssertionError, ValueError):
                caught.append(fn.__name__)
    assert caught, f"no pin caught the planted mistake {name}"


@pytest.mark.parametrize("name", sorted(MUTANTS_NEXT))
def test_planted_mistake_in_next_functions_is_caught(name, src_text, tmp_path):
    old, new = MUTANTS_NEXT[name]
    assert src_text.count(old) == 1, f"mutation anchor for {name} not unique"
    src = tmp_path / "mutant.c"
    src.write_text(src_text.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run([obuild._cc(), "-std=c99", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
                    str(src), "-o", str(lib), "-lm"], check=True)
    caught = []
    with oracle.use_library(str(lib)):
        for fn, kw in PIN_CALLS_NEXT:
            try:
                fn(**kw)
            except (AssertionError, ValueError):
                caught.append(fn.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
