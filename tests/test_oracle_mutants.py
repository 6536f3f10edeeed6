"""Planted mistakes in the oracle must be caught by its pins (CPU only).

Each case copies qmm_oracle.c, plants one plausible mistake (a dropped term, a
wrong sign, offset, index, bias or rounding rule), compiles the copy into a
temporary directory, swaps it in for the real oracle and runs the pins of
oracle_pins.py until one fails.  A mutant that passes every pin means the pins
have a hole.  The real oracle is never modified.
"""
import ctypes
import os
import subprocess
import tempfile

import pytest

import oracle as O
import oracle_pins as P

SRC = os.path.join(os.path.dirname(O.__file__), "qmm_oracle.c")

# (name, text to find, replacement, occurrence index or None for all)
MUTANTS = [
    ("q4_offset_7", "(double)(lo - 8)", "(double)(lo - 7)", None),
    ("q4_nibbles_swapped", "int lo = blk[2 + j] & 0x0F;\n      int hi = blk[2 + j] >> 4;",
     "int hi = blk[2 + j] & 0x0F;\n      int lo = blk[2 + j] >> 4;", None),
    ("q4_scale_sign", "amax_s / -8.0f", "amax_s / 8.0f", None),
    ("q4_round_trunc", "int qi = (int)roundf(t) + 8;", "int qi = (int)t + 8;", None),
    ("q4_amax_last_tie", "if (ax > amax) {", "if (ax >= amax) {", None),
    ("f16_subnormal_exp", "ldexp((double)m, -24); /* subnormal", "ldexp((double)m, -25); /* subnormal", None),
    ("f16_bias", "(double)m / 1024.0, e - 15)", "(double)m / 1024.0, e - 14)", None),
    ("bf16_shift", "(uint32_t)h << 16", "(uint32_t)h << 15", None),
    ("e4m3_bias", "(double)m / 8.0, e - 7)", "(double)m / 8.0, e - 8)", None),
    ("e4m3_subnormal", "ldexp((double)m, -9); /* subnormal", "ldexp((double)m, -10); /* subnormal", None),
    ("f16_encode_ties_away", "static double rne_int(double x) { return nearbyint(x); }",
     "static double rne_int(double x) { return round(x); }", None),
    ("e4m3_encode_no_sat", "if (a >= 448.0) return (uint8_t)(sign | 0x7Eu);",
     "if (a >= 480.0) return (uint8_t)(sign | 0x7Fu);", None),
    ("fp8_scale_448_to_240", "amax / 448.0f", "amax / 240.0f", None),
    ("fwht_sign_f32", "v[i + h] = x - y;", "v[i + h] = y - x;", 0),
    ("fwht_sign_f64", "v[i + h] = x - y;", "v[i + h] = y - x;", 1),
    ("fwht_missing_stage", "for (int h = 1; h < B; h <<= 1) {", "for (int h = 1; h < B / 2; h <<= 1) {", None),
    ("fwht_stage_order", "for (int h = 1; h < B; h <<= 1) {\n    for (int i = 0; i < B; ++i) {\n      if (i & h) continue;\n      float x",
     "for (int hh = B / 2; hh >= 1; hh >>= 1) { int h = hh;\n    for (int i = 0; i < B; ++i) {\n      if (i & h) continue;\n      float x", None),
    ("fwht_order_only_above_32", "for (int h = 1; h < B; h <<= 1) {\n    for (int i = 0; i < B; ++i) {\n      if (i & h) continue;\n      float x",
     "for (int hh = 1; hh < B; hh <<= 1) { int h = (B > 32 && hh >= 16) ? (hh == 16 ? B / 2 : hh / 2) : hh;\n    for (int i = 0; i < B; ++i) {\n      if (i & h) continue;\n      float x", None),
    ("h32_weights_not_divided", "r[j] = r[j] * 0.03125f;", "r[j] = r[j] * 0.0625f;", None),
    ("rotated_weights_scale", "r[j] = r[j] * inv_b;", "r[j] = r[j] * (2.0f * inv_b);", None),
    ("act_rotation_block_32", "const int B = hadamard == 1 ? 32 : hadamard;", "const int B = 32;", None),
    ("act_rotation_first_row_only", "  if (hadamard) {\n    for (int m = 0; m < M; ++m)",
     "  if (hadamard) {\n    for (int m = 0; m < 1; ++m)", None),
    ("product_drops_last_term", "          for (int64_t k = 0; k < K; ++k) {\n            double p = a[(int64_t)m * K + k] * w[k];",
     "          for (int64_t k = 0; k < K - 1; ++k) {\n            double p = a[(int64_t)m * K + k] * w[k];", None),
    ("product_sabs_signed", "            sabs += fabs(p);\n          }\n          out[(int64_t)m * nrows + i]",
     "            sabs += p;\n          }\n          out[(int64_t)m * nrows + i]", None),
    ("product_wrong_act_row", "double p = a[(int64_t)m * K + k] * w[k];", "double p = a[(int64_t)(M - 1 - m) * K + k] * w[k];", None),
    ("q8_codes_unsigned", "d * (double)(int8_t)blk[2 + j]", "d * (double)blk[2 + j]", None),
    ("q8_scale_128", "float d32 = amax / 127.0f;", "float d32 = amax / 128.0f;", None),
    ("q8_round_trunc", "int qi = (int)roundf(x[j] * inv);", "int qi = (int)(x[j] * inv);", None),
    ("q8_drops_sign_of_d", "(uint16_t)(blk[0] | (blk[1] << 8)));\n    for (int j = 0; j < 32; ++j) row",
     "(uint16_t)(blk[0] | ((blk[1] & 0x7F) << 8)));\n    for (int j = 0; j < 32; ++j) row", None),
    ("greedy_last_tie", "  return x > y;\n}", "  return x >= y;\n}", None),
    ("greedy_argmin", "  return x > y;\n}", "  return x < y;\n}", None),
    ("greedy_nan_ignored", "if (score_above(row[n], row[best])) best = n;", "if (row[n] > row[best]) best = n;", None),
    ("greedy_last_nan", "  if (isnan(y)) return 0;\n", "", None),
    ("greedy_token_offset", "argmax[k] == tokens[k + 1]", "argmax[k] == tokens[k]", None),
    ("greedy_k_short", "while (k < M - 1 && argmax", "while (k < M - 2 && argmax", None),
    ("greedy_next_is_last_draft", "result[1] = argmax[k];", "result[1] = argmax[k > 0 ? k - 1 : 0];", None),
    ("fp8_scale_tile_transposed", "double s = (double)scales[(n / 128) * tk_n + k / 128];",
     "double s = (double)scales[(n / 128) * tk_n + (k / 128 + n / 128) % tk_n];", None),
]


def _mutate(text, find, repl, occ):
    assert find in text, f"mutation anchor not found: {find!r}"
    if occ is None:
        return text.replace(find, repl)
    idx = -1
    for _ in range(occ + 1):
        idx = text.index(find, idx + 1)
    return text[:idx] + repl + text[idx + len(find):]


@pytest.mark.parametrize("name,find,repl,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, find, repl, occ, tmp_path):
    with open(SRC) as f:
        text = f.read()
    mutated = _mutate(text, find, repl, occ)
    assert mutated != text
    src = tmp_path / "mutant.c"
    src.write_text(mutated)
    so = tmp_path / "libmutant.so"
    r = subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                        "-fopenmp", str(src), "-o", str(so), "-lm"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    mutant = O._configure(ctypes.CDLL(str(so)))
    saved = O._lib
    O._lib = mutant
    caught = []
    try:
        for check in P.ALL_CHECKS:
            try:
                check(O)
            except AssertionError:
                caught.append(check.__name__)
                break
    finally:
        O._lib = saved
    assert caught, f"mutant {name} passed every pin"
