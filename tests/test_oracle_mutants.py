"""Plant plausible mistakes in copies of the oracle; the pins must catch each.

Every mutant is the oracle's own source with one textual change, compiled on
the CPU into a temporary library.  A mutant that passes every pin would mean
the pins cannot tell that mistake from the right answer.
"""
import os

import pytest

import oracle
from oracle_pins import PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.cpp")

MUTANTS = {
    "dropped_bias": ("const double w = (double)q * scale + bias;", "const double w = (double)q * scale;"),
    "bias_subtracted": ("const double w = (double)q * scale + bias;", "const double w = (double)q * scale - bias;"),
    "high_nibble_first": ("const int q = (int)((packed >> bit_offset) & 0xFu);",
                          "const int q = (int)((packed >> (28 - bit_offset)) & 0xFu);"),
    "code_at_high_nibble_first": ("return (int)((word >> (4 * (k % 8))) & 0xFu);",
                                  "return (int)((word >> (28 - 4 * (k % 8))) & 0xFu);"),
    "wrong_scale_group": ("const double scale = bf16_decode(S[n * groups + g]);",
                          "const double scale = bf16_decode(S[n * groups + (g + 1) % groups]);"),
    "activation_group_offset_dropped": ("xrow[g * G + p * 8 + bit_offset / 4]", "xrow[p * 8 + bit_offset / 4]"),
    "rows_swapped": ("dot_one(x + m * K, Wq,", "dot_one(x + (M - 1 - m) * K, Wq,"),
    "absdot_signed": ("abs_sum += std::fabs(a * w);", "abs_sum += a * w;"),
    "ties_away_from_zero": ("else r = (std::fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "else r = fl + 1.0;"),
    "truncation": ("if (diff > 0.5) r = fl + 1.0;", "if (diff > 2.0) r = fl + 1.0;"),
    "decode_exponent_bias": ("efield - 127 - 7", "efield - 127 - 6"),
    "wrong_expert": ("dot_one(x + t * K, Wq + e * words", "dot_one(x + t * K, Wq + (E - 1 - e) * words"),
    "dequant_scale_group": ("bf16_decode(S[n * groups + k / G]) +", "bf16_decode(S[n * groups]) +"),
    "group_size_fixed_at_64": ("const int64_t words_per_group = G / 8;", "const int64_t words_per_group = 8;"),
    "dequant_bias_group_halved": ("bf16_decode(B[n * groups + k / G]);", "bf16_decode(B[n * groups + k / G / 2]);"),
    # STQ1_0
    "stq1_zero_lane_from_low_bits": ("const int zero_lane = c >> 2;", "const int zero_lane = c & 3;"),
    "stq1_flip_bits_swapped": ("const int flip = rank == 0 ? (c & 1) : rank == 1 ? ((c >> 1) & 1) : 0;",
                               "const int flip = rank == 0 ? ((c >> 1) & 1) : rank == 1 ? (c & 1) : 0;"),
    "stq1_flip_reaches_last_lane": ("const int flip = rank == 0 ? (c & 1) : rank == 1 ? ((c >> 1) & 1) : 0;",
                                    "const int flip = rank == 2 ? (c & 1) : rank == 1 ? ((c >> 1) & 1) : 0;"),
    "stq1_group_sign_ignored": ("  if (s)\n    for (int l = 0; l < 4; ++l) v[l] = -v[l];", "  (void)s;"),
    "stq1_element_offset_map": ("const int g = (w / 64) * 16 + w % 16;\n  const int p = (w % 64) / 16;",
                                "const int g = w / 4;\n  const int p = w % 4;"),
    "stq1_lane_group_transposed": ("const int g = (w / 64) * 16 + w % 16;\n  const int p = (w % 64) / 16;",
                                   "const int g = (w / 64) * 16 + (w % 64) / 4;\n  const int p = w % 4;"),
    "stq1_high_nibble_first": ("(block[g / 2] >> (4 * (g % 2)))", "(block[g / 2] >> (4 - 4 * (g % 2)))"),
    "stq1_sign_bit_msb_first": ("(block[32 + g / 8] >> (g % 8))", "(block[32 + g / 8] >> (7 - g % 8))"),
    "stq1_scale_big_endian": ("(uint16_t)(block[40] | (block[41] << 8))", "(uint16_t)(block[41] | (block[40] << 8))"),
    "stq1_fp16_exponent_bias": ("efield - 15 - 10", "efield - 15 - 9"),
    "stq1_blocks_reversed": ("blocks + (n * nb + b) * kStqBytes", "blocks + (n * nb + (nb - 1 - b)) * kStqBytes"),
    "stq1_x_block_offset_dropped": ("xrow[b * kStqWeights + w]", "xrow[w]"),
    "stq1_wrong_expert": ("blocks + e * per_expert", "blocks + (E - 1 - e) * per_expert"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, f"mutation site for {name} not found exactly once"
    path = tmp_path / f"oracle_{name}.cpp"
    path.write_text(src.replace(before, after))
    lib = oracle.build(str(path), str(tmp_path / f"lib_{name}.so"), force=True)
    o = oracle.Oracle(oracle.load(lib))
    for pin in PINS:
        try:
            pin(o)
        except (AssertionError, ValueError, ZeroDivisionError, OverflowError):
            return  # caught
    pytest.fail(f"no pin catches the mutant {name}")
