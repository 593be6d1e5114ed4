"""The oracle pins must catch plausible mistakes.

Each case copies the oracle's C source to a temporary directory, plants one
mistake by a textual substitution, builds the copy and runs the pin suite
against it in a child process. Every mutant must make the pins fail. The
real oracle is never modified.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "awq_oracle.c")

MUTANTS = {
    "sign_of_q_minus_z": ("int d = (int)q[k * N + n] - (int)z[gi * N + n];",
                          "int d = (int)z[gi * N + n] - (int)q[k * N + n];"),
    "nibble_order_reversed": ("(w >> (4 * i)) & 0xFu", "(w >> (4 * (7 - i))) & 0xFu"),
    "group_index_modulo": ("int64_t gi = k / g;", "int64_t gi = k % (K / g);"),
    "scale_from_group_zero": ("awq_oracle_f16_to_f64(scales[gi * N + n])",
                              "awq_oracle_f16_to_f64(scales[n])"),
    "bias_dropped": ("j->y[r * N + j->n0 + n] = acc[n] + b;", "j->y[r * N + j->n0 + n] = acc[n];"),
    "first_k_term_dropped": ("for (int64_t k = 0; k < K; ++k) {\n            double xv",
                             "for (int64_t k = 1; k < K; ++k) {\n            double xv"),
    "ties_away_from_zero": ("return (fmod(r, 2.0) == 0.0) ? r : r + 1.0;", "return r + 1.0;"),
    "weights_transposed_read": ("const uint16_t *wrow = j->W16 + k * N + j->n0;",
                                "const uint16_t *wrow = j->W16 + (k % N) * N + j->n0;"),
    "pack_nibble_order_reversed": ("& 0xFu) << (4 * i);", "& 0xFu) << (4 * (7 - i));"),
    "quantize_ties_round_up": ("return (fmod(lo, 2.0) != 0.0) ? lo + 1.0 : lo;", "return lo + 1.0;"),
    "quantize_zero_point_dropped": ("int c = (int)round_half_even_signed(t) + (int)zrow[n];",
                                    "int c = (int)round_half_even_signed(t);"),
    "quantize_no_clamp": ("q[k * N + n] = (uint8_t)(c < 0 ? 0 : (c > 15 ? 15 : c));",
                          "q[k * N + n] = (uint8_t)c;"),
    "quantize_scale_of_group_zero": ("const uint16_t *srow = scales + grp * N;",
                                     "const uint16_t *srow = scales;"),
    "gidx_table_ignored": ("const int64_t row_group = g_idx[k];", "const int64_t row_group = k % G;"),
    "gidx_zero_of_wrong_row": ("int diff = (int)q[k * N + n] - (int)z[row_group * N + n];",
                               "int diff = (int)q[k * N + n] - (int)z[(k % G) * N + n];"),
    "f16_encode_truncates": ("double s = round_half_even(ldexp(a, 10 - expo));",
                             "double s = floor(ldexp(a, 10 - expo));"),
    "f16_decode_subnormal_as_normal": ("v = ldexp((double)frac, -24);",
                                       "v = ldexp((double)(1024 + frac), -25);"),
    "f16_encode_subnormal_scale": ("double m = round_half_even(ldexp(a, 24));",
                                   "double m = round_half_even(ldexp(a, 23));"),
    "zero_point_of_group_zero": ("int d = (int)q[k * N + n] - (int)z[gi * N + n];",
                                 "int d = (int)q[k * N + n] - (int)z[n];"),
    "sum_rounded_to_f16_before_bias": ("j->y[r * N + j->n0 + n] = acc[n] + b;",
                                       "j->y[r * N + j->n0 + n] = "
                                       "awq_oracle_f16_to_f64(awq_oracle_f64_to_f16(acc[n])) + b;"),
    "sampled_row_read_from_sample_index": ("double xv = awq_oracle_f16_to_f64(j->x[m * K + k]);",
                                           "double xv = awq_oracle_f16_to_f64(j->x[r * K + k]);"),
    "group_minus_one_rule_missing": ("int64_t g = (group_size == -1) ? in_features : group_size;",
                                     "int64_t g = group_size;"),
    "pack_keeps_high_bits": ("w |= (uint32_t)(codes[r * cols + 8 * j + i] & 0xFu) << (4 * i);",
                             "w |= (uint32_t)codes[r * cols + 8 * j + i] << (4 * i);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, f"mutation site for {name} not found exactly once"
    mutant = tmp_path / "awq_oracle_mutant.c"
    mutant.write_text(src.replace(before, after))
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                    "-pthread", str(mutant), "-o", str(lib), "-lm"], check=True)
    env = dict(os.environ, AWQ_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
