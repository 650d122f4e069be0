"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (on the CPU,
in a temporary directory), builds it, and runs the pin tests of
``test_oracle_pins`` against that build: at least one pin must fail.  The
real oracle is never modified.
"""
import os
import shutil
import tempfile

import pytest

from oracle import oracle as O
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(O.__file__), "fadkv_oracle.c")

# (name, original text, planted text)
MUTANTS = [
    ("drop lambda_abs", "lambda_abs + lambda_rel * Lwork[i * k + i]", "lambda_rel * Lwork[i * k + i]"),
    ("lambda_rel not scaled by G_ii", "lambda_abs + lambda_rel * Lwork[i * k + i]", "lambda_abs + lambda_rel"),
    ("residual sign", "acc -= c[i] * D[(int64_t)S[i] * d + t];", "acc += c[i] * D[(int64_t)S[i] * d + t];"),
    ("greedy tie to higher id", "(a == abest && P[i] < P[best])", "(a == abest && P[i] > P[best])"),
    ("top-n tie to higher id", "return (a->id < b->id) ? -1 : (a->id > b->id);", "return (a->id > b->id) ? -1 : (a->id < b->id);"),
    ("greedy correlates x instead of e", "double a = fabs(dot(D + (int64_t)P[i] * d, e, d));", "double a = fabs(dot(D + (int64_t)P[i] * d, x, d));"),
    ("Gram index slip", "double g = dot(D + (int64_t)S[i] * d, D + (int64_t)S[l] * d, d);", "double g = dot(D + (int64_t)S[i] * d, D + (int64_t)S[i] * d, d);"),
    ("screening without abs", "rk[j].mag = fabs(dot(D + (int64_t)j * d, x, d));", "rk[j].mag = dot(D + (int64_t)j * d, x, d);"),
    ("rhs uses the wrong atom", "bwork[i] = dot(D + (int64_t)S[i] * d, x, d);", "bwork[i] = dot(D + (int64_t)S[0] * d, x, d);"),
    ("back substitution transposed", "v -= Lwork[m * k + i] * c[m];", "v -= Lwork[i * k + m] * c[m];"),
    ("relres not relative", "relres[v] = (xn == 0.0) ? 0.0 : en / xn;", "relres[v] = en;"),
    ("adapt threshold not strict", "if (!(relres[v] > delta)) continue;", "if (!(relres[v] >= delta)) continue;"),
    ("adapt inactive order reversed", "for (int j = 0; j < N; ++j)\n        if (append ? usage[j] < 0 : usage[j] == 0) L[nL++] = j;", "for (int j = N - 1; j >= 0; --j)\n        if (append ? usage[j] < 0 : usage[j] == 0) L[nL++] = j;"),
    ("append mode reuses inactive atoms", "append ? usage[j] < 0 : usage[j] == 0", "append ? usage[j] <= 0 : usage[j] == 0"),
    ("fixed size takes free slots", "append ? usage[j] < 0 : usage[j] == 0", "append ? usage[j] < 0 : usage[j] <= 0"),
    ("adapt new atom usage stays 0", "usage[j] = 1;\n        repl_id[v] = j;", "repl_id[v] = j;"),
    ("adapt residual keeps first term only", "for (int k = 0; k < s; ++k) {\n                int32_t a = idx[(int64_t)v * s + k];\n                if (a >= 0)\n                    acc -=", "for (int k = 0; k < 1; ++k) {\n                int32_t a = idx[(int64_t)v * s + k];\n                if (a >= 0)\n                    acc -="),
    ("adapt repl_coef squared norm", "repl_coef[v] = en;", "repl_coef[v] = en * en;"),
    ("reconstruct drops replacement", "acc += repl_coef[v] * load_elem", "acc += 0.0 * load_elem"),
    ("half rounding truncates", "double q = nearbyint(ldexp(a, 10 - E));", "double q = floor(ldexp(a, 10 - E));"),
    ("half subnormal scale", "v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    ("pack truncates", "double q = nearbyint(ldexp(m, 11));", "double q = floor(ldexp(m, 11));"),
    ("pack exponent off by one", "int be = E - 1 + 127;", "int be = E + 127;"),
    ("attend scale dropped", "sc[t] = scale * dot(qh, kv, d);", "sc[t] = dot(qh, kv, d);"),
    ("attend head grouping", "const int hk = h / grp;", "const int hk = h % Hkv;"),
    ("attend skips the replacement word", "for (int i = 0; i < W; ++i) {\n                    uint32_t w = ck", "for (int i = 0; i + 1 < W; ++i) {\n                    uint32_t w = ck"),
    ("attend ignores lengths", "int T = lengths[b] < 0 ? 0 : (lengths[b] > Tmax ? Tmax : lengths[b]);", "int T = Tmax;"),
    ("PL takes ranks 1..s", "for (int k = 0; k < s; ++k) S[k] = rk[k].id;", "for (int k = 0; k < s; ++k) S[k] = rk[k + 1].id;"),
    ("PL ids left in rank order", "qsort(S, (size_t)s, sizeof(int32_t), cmp_i32);", ";"),
    ("PL residual drops the last atom", "for (int k = 0; k < s; ++k)\n                acc -= c[k]", "for (int k = 0; k + 1 < s; ++k)\n                acc -= c[k]"),
    ("PL relres squared norm", "sqrt(en2) / xn", "en2 / xn"),
    ("given pool read from vector 0", "P[i] = pool_in[(int64_t)v * n + i];", "P[i] = pool_in[i];"),
    ("given pool shifted by one", "P[i] = pool_in[(int64_t)v * n + i];", "P[i] = pool_in[(int64_t)v * n + i + (i + 1 < n)];"),
    ("given pool ignored", "        if (pool_in) {\n            for (int i = 0; i < n; ++i) {", "        if (0 && pool_in) {\n            for (int i = 0; i < n; ++i) {"),
]

PIN_TESTS = [
    pins.test_half_decode_exhaustive,
    pins.test_half_encode_rounding,
    pins.test_table4_cost_reproduced_by_operation_count,
    lambda O: pins.test_topn_matches_full_sort(O, 512, 64, 32, pins.np.float32),
    pins.test_topn_tie_rule_on_exact_zeros,
    pins.test_ridge_matches_normal_equations,
    pins.test_orthogonal_closed_form,
    pins.test_unit_orthonormal_relres_constant,
    lambda O: pins.test_exact_recovery_incoherent(O, False),
    pins.test_greedy_steps_brute_force,
    pins.test_brute_force_subset_objective,
    pins.test_greedy_on_pool_restricted_closed_form,
    pins.test_greedy_on_pool_matches_encode_and_ignores_order,
    pins.test_zero_and_nonfinite_inputs,
    pins.test_adapt_golden_cases,
    pins.test_adapt_invariants_random,
    pins.test_append_growth_against_fixed_size,
    pins.test_reconstruct_consistency,
    pins.test_table4_pl_cost_reproduced_by_operation_count,
    pins.test_pl_weighted_orthogonal_closed_form,
    lambda O: pins.test_pl_with_one_atom_is_the_first_greedy_pick(O, pins.np.float32),
    pins.test_pl_is_greedy_over_a_pool_of_s,
    pins.test_pl_fit_matches_normal_equations,
    pins.test_pl_zero_and_nonfinite_inputs,
    pins.test_pack_word_matches_binary16_rounding,
    pins.test_pack_word_layout,
    pins.test_attend_single_token_is_its_value,
    pins.test_attend_two_tokens_closed_form,
    pins.test_attend_grouped_heads_and_lengths,
    pins.test_attend_identical_keys_average_values,
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique/found: {name}"
    tmp = tempfile.mkdtemp(prefix="oracle_mutant_")
    try:
        path = os.path.join(tmp, "mutant.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        so = O.compile_source(path, os.path.join(tmp, "libmutant.so"), force=True)
        variant = O.Variant(so)
        caught = []
        for t in PIN_TESTS:
            try:
                t(variant)
            except (AssertionError, RuntimeError, ValueError, IndexError):
                caught.append(getattr(t, "__name__", "pin"))
                break
        assert caught, f"no pin caught the planted mistake: {name}"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
