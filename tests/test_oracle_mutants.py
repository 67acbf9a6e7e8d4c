"""Planted mistakes: each mutant is a copy of oracle.c with one plausible
error (a dropped term, a wrong sign, order or index, a different rounding),
compiled on the CPU.  The pins must catch every one of them; a mutant that
passes every pin would mean the pins cannot tell that mistake apart."""
import os

import pytest

import oracle
from oracle_pins import PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "reverse_rank_order": (
        "for (int r = 1; r < W; ++r)\n        acc = acc + oracle_bf16_to_f32(x[r][idx]);",
        "for (int r = W - 1; r >= 1; --r)\n        acc = acc + oracle_bf16_to_f32(x[r][idx]);"),
    "seed_with_positive_zero": (
        "float acc = oracle_bf16_to_f32(x[0][idx]);\n    for (int r = 1;",
        "float acc = 0.0f;\n    for (int r = 0;"),
    "subtract_partial": (
        "acc = acc + oracle_bf16_to_f32(x[r][idx]);",
        "acc = acc - oracle_bf16_to_f32(x[r][idx]);"),
    "wrong_partial_index": (
        "acc = acc + oracle_bf16_to_f32(x[r][idx]);",
        "acc = acc + oracle_bf16_to_f32(x[0][idx]);"),
    "drop_residual": (
        "oracle_bf16_to_f32(reduced[i]) + oracle_bf16_to_f32(residual[i])",
        "oracle_bf16_to_f32(reduced[i])"),
    "ties_away_from_zero": (
        "(dropped == 0x8000u && (kept & 1u))", "(dropped == 0x8000u)"),
    "truncate_instead_of_round": (
        "kept += 1u;", "kept += 0u;"),
    "nan_not_quieted": (
        "return (uint16_t)(kept | 0x0040u);", "return (uint16_t)kept;"),
    "eps_outside_root": (
        "1.0f / sqrtf(mean + eps)", "1.0f / (sqrtf(mean) + eps)"),
    "no_division_by_H": (
        "float mean = ss / (float)H;", "float mean = ss;"),
    "sum_not_squared": (
        "ss = ss + v * v;", "ss = ss + v;"),
    "weight_dropped": (
        "oracle_f32_to_bf16(n * oracle_bf16_to_f32(weight[h]))",
        "oracle_f32_to_bf16(n)"),
    "weight_index_fixed": (
        "oracle_bf16_to_f32(weight[h])", "oracle_bf16_to_f32(weight[0])"),
    "divide_instead_of_multiply": (
        "float n = v * rstd;", "float n = v / rstd;"),
    "row_offset_wrong": (
        "int64_t off = t * H;\n        for (int r = 0; r < W; ++r)\n            row_x[r] = x[r] + off;\n        oracle_rank_sum(row_x",
        "int64_t off = t * (H - 1);\n        for (int r = 0; r < W; ++r)\n            row_x[r] = x[r] + off;\n        oracle_rank_sum(row_x"),
    "f32_partials_prerounded": (
        "acc = acc + x[r][idx];",
        "acc = acc + oracle_bf16_to_f32(oracle_f32_to_bf16(x[r][idx]));"),
    "f32_reverse_rank_order": (
        "for (int r = 1; r < W; ++r)\n        acc = acc + x[r][idx];",
        "for (int r = W - 1; r >= 1; --r)\n        acc = acc + x[r][idx];"),
    "f32_first_partial_dropped": (
        "float acc = x[0][idx];", "float acc = 0.0f * x[0][idx];"),
    "f32_row_offset_wrong": (
        "            row_x[r] = x[r] + off;\n        oracle_rank_sum_f32",
        "            row_x[r] = x[r] + off / 2;\n        oracle_rank_sum_f32"),
    "e4m3_overflow_to_nan": (
        "return (uint8_t)(sign | 0x7Eu);          /* saturate to 448 */",
        "return (uint8_t)(sign | 0x7Fu);          /* saturate to 448 */"),
    "e4m3_truncates": ("float k = rintf(a / step);", "float k = truncf(a / step);"),
    "e4m3_wrong_bias": ("(uint8_t)((E + 7) << 3)", "(uint8_t)((E + 8) << 3)"),
    "quant_scale_wrong_max": ("amax / 448.0f : 1.0f", "amax / 240.0f : 1.0f"),
    "quant_uses_scale_not_inverse": ("oracle_bf16_to_f32(norm[h]) * inv)", "oracle_bf16_to_f32(norm[h]) * scale)"),
    "quant_inverse_off": ("448.0f / amax : 1.0f", "440.0f / amax : 1.0f"),
    "quant_amax_signed": ("float v = fabsf(oracle_bf16_to_f32(norm[h]));", "float v = oracle_bf16_to_f32(norm[h]);"),
    "combine_fused_multiply_add": (
        "        acc = acc + prod;",
        "        acc = fmaf(gates_row[k], oracle_bf16_to_f32(expert_out[(int64_t)s * H + h]), acc);"),
    "combine_gate_index_wrong": ("gates_row[k] * oracle", "gates_row[0] * oracle"),
    "combine_no_range_check": ("if (s < 0 || (int64_t)s >= n_slots)", "if (s < 0)"),
    "combine_slot_row_wrong": ("expert_out[(int64_t)s * H + h]", "expert_out[(int64_t)s + h]"),
    "e2m1_ties_away": ("float v = rintf(a / step) * step;", "float v = roundf(a / step) * step;"),
    "e2m1_wrong_bias": ("(uint8_t)((E + 1) << 1)", "(uint8_t)((E + 2) << 1)"),
    "nvfp4_nibbles_swapped": ("(uint8_t)(lo | (hi << 4))", "(uint8_t)(hi | (lo << 4))"),
    "nvfp4_half_block_amax": ("for (int i = 0; i < 16; ++i) {", "for (int i = 0; i < 8; ++i) {"),
    "nvfp4_tensor_scale_inverted": ("float inv = sv > 0.0f ? g / sv : 0.0f;",
                                    "float inv = sv > 0.0f ? 1.0f / (sv * g) : 0.0f;"),
    "nvfp4_scale_without_tensor_scale": ("oracle_f32_to_e4m3_sat((amax / 6.0f) * g)",
                                         "oracle_f32_to_e4m3_sat(amax / 6.0f)"),
    "widen_drops_low_bit": (
        "uint32_t u = ((uint32_t)b) << 16;", "uint32_t u = ((uint32_t)(b & 0xFFFEu)) << 16;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site for {name} not found exactly once"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new))
    lib = oracle.load_library(oracle.compile_oracle(str(src), str(tmp_path / "libmutant.so")))
    O = oracle.Oracle(lib)
    caught = []
    for pin in PINS:
        try:
            pin(O)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
