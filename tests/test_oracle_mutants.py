"""Planted mistakes in a copy of the oracle must each fail at least one pin.

Each mutant is a one-line textual change to a temporary copy of oracle.c
(a dropped term, a wrong sign, index or bit order, a transposed operand, a
wrong rounding rule), compiled with gcc on the CPU and run through the same
pins as the real oracle.  A mutant that passes every pin would mean the pins
cannot tell that mistake from the method.
"""
import os
import shutil

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "key_includes_sign": ("unsigned key_i = row[g0 + i] & 0x7FFFu;",
                          "unsigned key_i = row[g0 + i] & 0xFFFFu;"),
    "ties_to_higher_column": ("< key_i)", "<= key_i)"),
    "mask_bit_order_msb_first": ("mrow[c / 32] |= 1u << (c % 32);",
                                 "mrow[c / 32] |= 1u << (31 - c % 32);"),
    "keeps_wrong_ranks": ("for (int k = 0; k < N; ++k) {", "for (int k = 1; k <= N; ++k) {"),
    "values_reversed_in_word": ("vrow[16 * w + k] = row[32 * w + b];",
                                "vrow[16 * w + 15 - k] = row[32 * w + b];"),
    "unpack_value_swap": ("out[32 * w + b] = vrow[16 * w + k];",
                          "out[32 * w + b] = vrow[16 * w + (k ^ 1)];"),
    "dot_drops_sign_of_x": ("acc += w * xc;", "acc += w * fabs(xc);"),
    "dot_reversed_x": ("double xc = orc_f16_to_f64(x[c]);",
                       "double xc = orc_f16_to_f64(x[cols - 1 - c]);"),
    "dot_drops_first_term": ("for (int64_t c = 0; c < cols; ++c) {",
                             "for (int64_t c = 1; c < cols; ++c) {"),
    "scale_signed": ("mag += fabs(w) * fabs(xc);", "mag += w * fabs(xc);"),
    "subnormal_scale": ("mag = ldexp((double)frac, -24);", "mag = ldexp((double)frac, -25);"),
    "normal_exponent_bias": ("ldexp((double)(1024 + frac), expo - 25)",
                             "ldexp((double)(1024 + frac), expo - 24)"),
    "ties_away_from_zero": ("return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "return fl + 1.0;"),
    "overflow_threshold": ("if (a >= 65520.0)", "if (a >= 65504.0)"),
    "bad_word_count_one_sided": ("if (popcount32(masks[i]) != 16) ++bad;",
                                 "if (popcount32(masks[i]) > 16) ++bad;"),
    "matvec_ignores_ld": ("dot_row(W + r * ld, x, cols,", "dot_row(W + r * cols, x, cols,"),
    "spmv_rows_ignores_ids": ("int64_t r = row_ids[i];", "int64_t r = i;"),
    "silu_sign": ("double silu = g[i] / (1.0 + exp(-g[i]));",
                  "double silu = g[i] / (1.0 + exp(g[i]));"),
    "silu_mul_drops_up": ("h[i] = silu * u[i];", "h[i] = silu;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation site for {name} not found"
    shutil.copy(os.path.join(os.path.dirname(SRC), "oracle.h"), tmp_path / "oracle.h")
    src = tmp_path / "oracle_mut.c"
    src.write_text(text.replace(old, new, 1))
    lib_path = oracle.build(str(src), str(tmp_path / "liboracle_mut.so"))
    mutant = oracle.Oracle(oracle.load(lib_path))
    failures = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError) as e:  # ValueError: rejected input
            failures.append(pin.__name__)
    assert failures, f"mutant {name} passed every pin"
