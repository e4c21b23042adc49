"""Plant plausible mistakes in copies of the CPU oracle and check that the pins catch each one.

Every mutant is one textual edit of ``oracle/h2o_oracle.c`` compiled into a temporary library; the
real source is never touched. A mutant that passes every pin would mean the pins cannot tell that
mistake from the method, so the test fails. Each edit must match the source exactly once, so a
refactor of the oracle that moves a mutated expression fails loudly here instead of silently
testing nothing.
"""

import os

import pytest

import oracle
import oracle_pins

MUTANTS = {
    "drop_sqrt_d_prefill": ("  const double scale = 1.0 / sqrt((double)D);\n\n  double* c",
                            "  const double scale = 1.0;\n\n  double* c"),
    "drop_sqrt_d_decode": ("  const double scale = 1.0 / sqrt((double)D);\n\n  /* Every unit",
                           "  const double scale = 1.0;\n\n  /* Every unit"),
    "row_sums_not_column_sums": ("for (int32_t j = 0; j <= i; ++j) c[j] += exp(s[j] - m) / l;",
                                 "for (int32_t j = 0; j <= i; ++j) c[i] += exp(s[j] - m) / l;"),
    "prefill_keeps_smallest": ("  if (x->c > y->c) return -1;\n  if (x->c < y->c) return 1;",
                               "  if (x->c > y->c) return 1;\n  if (x->c < y->c) return -1;"),
    "prefill_tie_keeps_earlier": ("return (x->pos > y->pos) ? -1 : (x->pos < y->pos) ? 1 : 0;",
                                  "return (x->pos < y->pos) ? -1 : (x->pos > y->pos) ? 1 : 0;"),
    "prefill_window_off_by_one": ("for (int32_t p = P - k_local; p < P; ++p) keep[p] = 1;",
                                  "for (int32_t p = P - k_local + 1; p < P; ++p) keep[p] = 1;"),
    "new_token_not_in_normaliser": ("for (int32_t j = 0; j <= n; ++j) l += exp(s[j] - m);",
                                    "for (int32_t j = 0; j < n; ++j) l += exp(s[j] - m);"),
    "new_token_not_in_output": ("      acc += p[n] * elem(v_new, dtype, (size_t)u * D + d);\n", "\n"),
    "no_accumulation": ("      sc[j] = sc[j] + add;", "      sc[j] = add;"),
    "evict_highest_score": ("if (best < 0 || sc[j] < sc[best] || (sc[j] == sc[best] && sp[j] < sp[best])) {",
                            "if (best < 0 || sc[j] > sc[best] || (sc[j] == sc[best] && sp[j] < sp[best])) {"),
    "tie_evicts_latest": ("if (best < 0 || sc[j] < sc[best] || (sc[j] == sc[best] && sp[j] < sp[best])) {",
                          "if (best < 0 || sc[j] < sc[best] || (sc[j] == sc[best] && sp[j] > sp[best])) {"),
    "protect_one_more": ("const int64_t last_candidate = (int64_t)t - k_local;",
                         "const int64_t last_candidate = (int64_t)t - k_local - 1;"),
    "protect_one_less": ("const int64_t last_candidate = (int64_t)t - k_local;",
                         "const int64_t last_candidate = (int64_t)t - k_local + 1;"),
    "new_score_zero": ("    sc[target] = (float)p[n];", "    sc[target] = 0.0f;"),
    "wrong_position_written": ("    sp[target] = t;", "    sp[target] = t - 1;"),
    "evict_before_accumulate": ("      float add = (float)p[j];", "      float add = 0.0f;"),
    "topk_accumulates": ("        sc[j] = add;  /* Top-K ranks by the current step's attention only */",
                         "        sc[j] = sc[j] + add;"),
    "topk_prefill_ranks_by_colsum": ("const double* start = pol->kind == H2O_ORACLE_POLICY_TOPK ? a : c;",
                                     "const double* start = c;"),
    "sink_off_by_one": ("case H2O_ORACLE_POLICY_SINK_WINDOW: return pos >= pol->n_sink;",
                        "case H2O_ORACLE_POLICY_SINK_WINDOW: return pos > pol->n_sink;"),
    "strided_grid_inverted": ("if (pol->kind == H2O_ORACLE_POLICY_STRIDED && pos % pol->stride == 0) return",
                              "if (pol->kind == H2O_ORACLE_POLICY_STRIDED && pos % pol->stride != 0) return"),
    "local_evicts_newest": ("if (best < 0 || position_rank(pol, sp[j]) < position_rank(pol, sp[best])) best = j;",
                            "if (best < 0 || position_rank(pol, sp[j]) > position_rank(pol, sp[best])) best = j;"),
    "attention_drops_sqrt_d": ("  const double scale = 1.0 / sqrt((double)D);\n  const size_t eb",
                               "  const double scale = 1.0;\n  const size_t eb"),
    "attention_unnormalised": ("acc += w[j] / l * elem(vu, dtype", "acc += w[j] * elem(vu, dtype"),
    "attention_skips_diagonal": ("for (int32_t j = 0; j <= i; ++j) acc += w[j] / l",
                                 "for (int32_t j = 0; j < i; ++j) acc += w[j] / l"),
    "attention_values_from_keys": ("acc += w[j] / l * elem(vu, dtype", "acc += w[j] / l * elem(ku, dtype"),
    "e4m3_ties_away_from_zero": ("double r = nearbyint(a / quantum) * quantum;",
                                 "double r = round(a / quantum) * quantum;"),
    "e4m3_no_saturation": ("  if (r > 448.0) r = 448.0;                     /* saturate */\n", "\n"),
    "e4m3_subnormal_spacing": ("if (binade < -6) binade = -6;", "if (binade < -7) binade = -7;"),
    "e4m3_scale_127": ("amax > 0.0f ? amax / 448.0f : 1.0f", "amax > 0.0f ? amax / 127.0f : 1.0f"),
    "e4m3_read_ignores_scale": ("return (double)c->scales[j] * e4m3_value(", "return 1.0 * e4m3_value("),
    "e4m3_exponent_bias": ("v = ldexp(8.0 + m, e - 10);", "v = ldexp(8.0 + m, e - 11);"),
    "new_value_row_from_key": ("store_row(&vc, (size_t)target, v_new, dtype, (size_t)u);",
                               "store_row(&vc, (size_t)target, k_new, dtype, (size_t)u);"),
}


@pytest.fixture(scope="module")
def source():
    with open(oracle.SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, source, tmp_path):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, f"mutation site for {name} not found exactly once"
    src = tmp_path / "h2o_oracle.c"
    src.write_text(source.replace(old, new))
    (tmp_path / "h2o_oracle.h").write_text(open(os.path.join(oracle.HERE, "h2o_oracle.h")).read())
    lib = oracle.build(str(src), str(tmp_path / f"lib_{name}.so"))
    caught = []
    for pin in oracle_pins.PINS:
        try:
            pin(lib)
        except Exception:  # any failure, incl. a pin crashing on nonsense state
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name!r}"
