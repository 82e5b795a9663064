"""Planted mistakes in copies of the oracle must each fail at least one pin.

Each mutant is the oracle's own C source with one plausible slip written in
(a wrong scale, a dropped or misplaced term, a swapped operand, a wrong stride,
a flipped sign, a missing guard).  The copies are compiled on the CPU into a
temporary directory; the real oracle is never modified.
"""
import pytest

import oracle
from oracle_pins import PINS

MUTANTS = [
    ("scale_1_over_D", "1.0 / sqrt((double)D)", "1.0 / (double)D"),
    ("unscaled_scores", "double s = dot * scale;", "double s = dot;"),
    ("normaliser_drops_max", "z += exp(scores[j - j0] - m);", "z += exp(scores[j - j0]);"),
    ("weights_unnormalised", "const double p = exp(scores[j - j0] - lse);",
     "const double p = exp(scores[j - j0] - m);"),
    ("values_from_keys", "const double *v_row = v_bh + j * (long long)D;",
     "const double *v_row = k_bh + j * (long long)D;"),
    ("scores_against_values", "const double *k_row = k_bh + j * (long long)D;",
     "const double *k_row = v_bh + j * (long long)D;"),
    ("head_stride_wrong",
     "k + bh * S * (long long)D,\n                 v + bh * S * (long long)D, j0, j1, D, scores,\n"
     "                 out + r * (long long)D",
     "k + bh * (long long)D,\n                 v + bh * (long long)D, j0, j1, D, scores,\n"
     "                 out + r * (long long)D"),
    ("merge_weight_sign", "const double wgt = exp(l - lse);", "const double wgt = exp(lse - l);"),
    ("merge_normaliser_drops_max", "z += exp(l - m);", "z += exp(l);"),
    ("merge_reads_empty_chunk",
     "      if (l == -INFINITY) continue;\n      const double wgt",
     "      const double wgt"),
    ("cfg_sign", "out[i] = eps_u[i] + w * (eps_c[i] - eps_u[i]);",
     "out[i] = eps_u[i] + w * (eps_u[i] - eps_c[i]);"),
    ("cfg_base", "out[i] = eps_u[i] + w * (eps_c[i] - eps_u[i]);",
     "out[i] = eps_c[i] + w * (eps_c[i] - eps_u[i]);"),
    ("key_range_off_by_one", "for (long long j = j0; j < j1; ++j) z +=",
     "for (long long j = j0 + 1; j < j1; ++j) z +="),
    ("relmae_base_of_cond", "base += fabs(eps_u[i]);", "base += fabs(eps_c[i]);"),
    ("relmae_signed_difference", "diff += fabs(d);", "diff += d;"),
    ("relmae_difference_of_base", "diff += fabs(d);", "diff += fabs(eps_u[i]);"),
    ("relmae_combine_sign", "out[i] = eps_u[i] + w * d;", "out[i] = eps_u[i] - w * d;"),
    ("relmae_ratio_inverted", "sums[2] = diff / base;", "sums[2] = base / diff;"),
    ("relmae_zero_base_finite", "diff == 0.0 ? 0.0 : INFINITY;", "0.0;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, old, new, tmp_path):
    src = oracle.source()
    assert src.count(old) == 1, f"mutation site for {name} not unique in the oracle"
    mutant = oracle.load_variant(src.replace(old, new), str(tmp_path))
    failed = []
    for pin in PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutant {name}"
