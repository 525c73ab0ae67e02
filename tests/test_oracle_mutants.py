"""Planted mistakes in a copy of the oracle must each fail at least one pin.

Each mutant below is a plausible slip (a dropped term, a wrong sign or index,
a transposed operand, the wrong reading of a garbled formula).  The mutant is
written to a temporary C file, compiled with the same flags as the oracle and
run through every check in _pins.py on the CPU.  A mutant that passes every
pin would mean the pins cannot tell that mistake from the real oracle.
"""
import os

import pytest

import _pins
import oracle

SRC = os.path.join(os.path.dirname(os.path.abspath(oracle.__file__)), "retention_oracle.c")

MUTANTS = {
    "gamma_1_based": ("return 1.0 - pow(2.0, -5.0 - (double)h);",
                      "return 1.0 - pow(2.0, -6.0 - (double)h);"),
    "parallel_not_causal": ("row[m] = (n >= m) ?", "row[m] = (1) ?"),
    "parallel_decay_sign": ("row[m] = (n >= m) ? pow(g, (double)(n - m))",
                            "row[m] = (n >= m) ? pow(g, (double)(m - n))"),
    "parallel_no_scale": ("dot(Q + (size_t)n * dk, K + (size_t)m * dk, dk) * scale",
                          "dot(Q + (size_t)n * dk, K + (size_t)m * dk, dk)"),
    "rows_decay_off_by_one": ("double w = pow(g, (double)(n - m)) *",
                              "double w = pow(g, (double)(n - m + 1)) *"),
    "recurrent_no_decay": ("S[(size_t)i * dv + j] = g * S[(size_t)i * dv + j] + kn[i] * vn[j];",
                           "S[(size_t)i * dv + j] = S[(size_t)i * dv + j] + kn[i] * vn[j];"),
    "recurrent_no_scale": ("s += qn[i] * scale * S[(size_t)i * dv + j];",
                           "s += qn[i] * S[(size_t)i * dv + j];"),
    "recurrent_transposed_outer": ("+ kn[i] * vn[j];", "+ kn[j % dk] * vn[i % dv];"),
    "chunk_zeta_off_by_one": ("const double zeta = pow(g, (double)(j + 1));",
                              "const double zeta = pow(g, (double)(j));"),
    "chunk_no_inner_decay_in_carry": ("const double w = pow(g, (double)(L - 1 - l));",
                                      "const double w = 1.0;"),
    "chunk_carry_full_chunk_on_tail": ("const double gL = pow(g, (double)L);",
                                       "const double gL = pow(g, (double)C);"),
    "chunk_inner_transposed": ("dot(qj, K + (size_t)(s + l) * dk, dk) * scale;",
                               "dot(Q + (size_t)(s + l) * dk, K + (size_t)(s + j) * dk, dk) * scale;"),
    "chunk_cross_term_dropped": ("oj[c] += zeta * scale * t;", "oj[c] += 0.0 * t;"),
    "groupnorm_unbiased_variance": ("var /= dv;", "var /= (dv - 1);"),
    "groupnorm_eps_outside_root": ("1.0 / sqrt(var + eps);", "1.0 / (sqrt(var) + eps);"),
    "groupnorm_weight_of_head_0": ("weight[h * dv + c]", "weight[c]"),
    "rotate_sine_sign": ("yr[2 * j] = xr[2 * j] * c - xr[2 * j + 1] * s;",
                         "yr[2 * j] = xr[2 * j] * c + xr[2 * j + 1] * s;"),
    "rotate_start_ignored": ("const double a = (double)(n0 + n) * theta[j];",
                             "const double a = (double)n * theta[j];"),
    "rotate_pairs_split": ("yr[2 * j + 1] = xr[2 * j] * s + xr[2 * j + 1] * c;",
                           "yr[2 * j + 1] = xr[(2 * j + 2) % d] * s + xr[2 * j + 1] * c;"),
    "bwd_dq_zeta_off_by_one": ("const double z = scale * pow(g, (double)(n + 1));",
                               "const double z = scale * pow(g, (double)n);"),
    "bwd_dq_decay_off_by_one": ("const double w = scale * pow(g, (double)(n - m)) *",
                                "const double w = scale * pow(g, (double)(n - m + 1)) *"),
    "bwd_dk_final_state_term_dropped": ("rk[i] += xi * dot(dS + (size_t)i * dv, V + (size_t)m * dv, dv);",
                                        "rk[i] += 0.0 * xi;"),
    "bwd_dv_scores_transposed": ("const double wv = d * dot(Q + (size_t)n * dk, K + (size_t)m * dk, dk);",
                                 "const double wv = d * dot(Q + (size_t)m * dk, K + (size_t)n * dk, dk);"),
    "bwd_no_scale_on_key_value_grads": ("const double d = scale * pow(g, (double)(n - m));",
                                        "const double d = pow(g, (double)(n - m));"),
    "bwd_ds0_no_decay_of_ds": ("double t = dS ? pow(g, (double)N) * dS[(size_t)i * dv + c] : 0.0;",
                               "double t = dS ? dS[(size_t)i * dv + c] : 0.0;"),
    "bwd_dv_final_state_transposed": ("for (int i = 0; i < dk; ++i) t += K[(size_t)m * dk + i] * dS[(size_t)i * dv + c];",
                                      "for (int i = 0; i < dk; ++i) t += K[(size_t)m * dk + i] * dS[(size_t)((i + c) % dk) * dv + c];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = oracle.build(force=True, src=str(path), out=str(tmp_path / f"{name}.so"))
    mutant = oracle.Oracle(lib)
    failed = []
    for check in _pins.ALL_CHECKS:
        try:
            check(mutant)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"mutant {name} passed every pin"
