"""Plant one mistake at a time in a copy of the oracle (on the CPU) and check
that the pin suite rejects every mutant.  Each mutant runs the pins in its own
process, so a mutant that reads out of bounds cannot take this run down."""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "drop_first_term": ("for (int64_t k = 0; k < K; ++k)", "for (int64_t k = 1; k < K; ++k)"),
    "wrong_sign": ("    for (int64_t k = 0; k < K; ++k)\n        s += oracle_half_to_double(a_row[k])",
                   "    for (int64_t k = 0; k < K; ++k)\n        s -= oracle_half_to_double(a_row[k])"),
    "f16acc_wrong_sign": ("k < k0 + 16 && k < j->K; ++k)\n                    s += ",
                          "k < k0 + 16 && k < j->K; ++k)\n                    s -= "),
    "transposed_result": ("dot_row_row(j->A + i * j->K, j->B + n * j->K, j->K)",
                          "dot_row_row(j->A + (n % j->M) * j->K, j->B + (i % j->N) * j->K, j->K)"),
    "b_row_from_i": ("j->B + n * j->K, j->K)", "j->B + (i % j->N) * j->K, j->K)"),
    "float_accumulator": ("    double s = 0.0;\n    for (int64_t k = 0; k < K; ++k)",
                          "    float s = 0.0f;\n    for (int64_t k = 0; k < K; ++k)"),
    "scaled_float_accumulator": ("            double s = 0.0;\n            for (int64_t k = 0; k < j->K; ++k) {",
                                 "            float s = 0.0f;\n            for (int64_t k = 0; k < j->K; ++k) {"),
    "round_via_float": ("j->D[i * j->N + n] = oracle_double_to_half(\n                dot_row_row(",
                        "j->D[i * j->N + n] = oracle_double_to_half((float)\n                dot_row_row("),
    "ties_to_odd": ("fmod(r, 2.0) != 0.0", "fmod(r, 2.0) == 0.0"),
    "truncate": ("if (rem > 0.5 || (rem == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;", ""),
    "subnormal_edge": ("(e_unb < -14 ? -14 : e_unb) - 10", "(e_unb < -15 ? -15 : e_unb) - 10"),
    "overflow_edge": ("if (a >= 65520.0)", "if (a >= 65504.0)"),
    "exponent_bias": ("expo - 25); /* 1.frac", "expo - 24); /* 1.frac"),
    "stages_floor": ("+ (copy_cycles % compute_cycles != 0);", ";"),
    "stages_no_plus_one": ("return in_flight + 1;", "return in_flight;"),
    "scaled_drop_beta": ("if (j->beta != 0.0) v += j->beta * oracle_half_to_double(j->C[i * j->N + n]);", ""),
    "scaled_alpha_skipped": ("double v = j->alpha * s;", "double v = s;"),
    "scaled_nn_read_as_tn": ("j->b_kn ? j->B[k * j->N + n] : j->B[n * j->K + k]",
                             "j->b_kn ? j->B[(n * j->K + k) % (j->K * j->N)] : j->B[n * j->K + k]"),
    "f16acc_slice_32": ("for (int64_t k0 = 0; k0 < j->K; k0 += 16) {", "for (int64_t k0 = 0; k0 < j->K; k0 += 32) {"),
    "f16acc_inner_32": ("k < k0 + 16 && k < j->K", "k < k0 + 32 && k < j->K"),
    "f16acc_no_slice_rounding": ("acc = oracle_half_to_double(oracle_double_to_half(s));", "acc = s;"),
    "scaled_beta_on_alpha": ("v += j->beta * oracle_half_to_double", "v += j->alpha * oracle_half_to_double"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    lib = oracle.compile_variant(src.replace(old, new), str(tmp_path / f"mut_{name}.so"))
    env = dict(os.environ, ORACLE_LIBRARY=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
