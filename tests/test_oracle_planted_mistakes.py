"""Each plausible mistake planted in a copy of the oracle source must fail at
least one of the oracle's pins (so the pins really constrain the oracle).

The mistakes are planted by text substitution in a temporary copy of
``oracle/moe_oracle.cpp`` compiled on the CPU; the oracle itself is untouched.
"""
import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
import test_oracle_finalize as tf
import test_oracle_index as ti
import test_oracle_permute as tp
import test_oracle_exp as tex
import test_oracle_route as tr
import test_oracle_scales as tsc
import test_oracle_sigmoid as tsg
import test_oracle_softmax as tsm

ORACLE_SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.cpp")

MUTANTS = {
    "group score = top-1 only": (
        "g[j] = (S == 1) ? group_vals[0] : group_vals[0] + group_vals[1];",
        "g[j] = group_vals[0];"),
    "group ties to the higher index": (
        "if (g[x] != g[y]) return g[x] > g[y];\n      return x < y;",
        "if (g[x] != g[y]) return g[x] > g[y];\n      return x > y;"),
    "expert ties to the higher index": (
        "if (b[x] != b[y]) return b[x] > b[y];\n      return x < y;",
        "if (b[x] != b[y]) return b[x] > b[y];\n      return x > y;"),
    "groups kept in index order": (
        "const int32_t j = group_order[m];", "const int32_t j = m;"),
    "bias kept in the weights": ("w[k] = s[allowed[k]];", "w[k] = b[allowed[k]];"),
    "normalisation dropped": ("w[k] = w[k] / sum;", "w[k] = w[k];"),
    "scale applied twice": ("w[k] = w[k] / sum;", "w[k] = w[k] / sum * scale;"),
    "bias subtracted": ("b[e] = s[e] + bias[e];", "b[e] = s[e] - bias[e];"),
    "unstable placement (reverse walk)": (
        "for (int64_t i = 0; i < N; ++i) {\n    const uint32_t pos",
        "for (int64_t i = N - 1; i >= 0; --i) {\n    const uint32_t pos"),
    "restore transposed": ("restore_token_order[i] = pos;", "restore_token_order[pos] = i;"),
    "CSR tail left at zero": ("expert_start_indices[j] = static_cast<uint32_t>(N);",
                              "expert_start_indices[j] = 0;"),
    "stats swapped": ("expert_usage_stats[0] = max_count;\n  expert_usage_stats[1] = active;",
                      "expert_usage_stats[0] = active;\n  expert_usage_stats[1] = max_count;"),
    "finalize drops the first term": (
        "for (int32_t k = 0; k < K; ++k) {\n      const int64_t row = restore[t * K + k];\n"
        "      acc = std::fma",
        "for (int32_t k = 1; k < K; ++k) {\n      const int64_t row = restore[t * K + k];\n"
        "      acc = std::fma"),
    "finalize restore indexed k-major": (
        "const int64_t row = restore[t * K + k];\n      acc = std::fma(w[t * K + k]",
        "const int64_t row = restore[k * T + t];\n      acc = std::fma(w[t * K + k]"),
    "finalize weight indexed k-major": (
        "acc = std::fma(w[t * K + k], bf16", "acc = std::fma(w[k * T + t], bf16"),
    "finalize reads down transposed": ("down[row * H + h]), acc)", "down[h * T * K + row]), acc)"),
    "scale offsets not rounded up": (
        "offset += (count[e] + row_align - 1) / row_align * row_align;",
        "offset += count[e] / row_align * row_align;"),
    "sigmoid drops a Taylor term": ("for (int k = 6; k >= 0; --k) p = std::fma(p, r, inv_fact[k]);",
                                    "for (int k = 6; k >= 1; --k) p = std::fma(p, r, inv_fact[k]);"),
    "sigmoid without the ln2 tail": ("r = std::fma(-n, 1.42860682030941723e-6f, r);", "r = r;"),
    "permute takes slot modulo K": ("const int64_t t = slot / K;", "const int64_t t = slot % K;"),
    "softmax without the max shift": ("ex[e] = exp_cody_waite(row[e] - m);",
                                      "ex[e] = exp_cody_waite(row[e]);"),
    "softmax sum skips the first expert": ("      sum += ex[e];", "      if (e > 0) sum += ex[e];"),
    "softmax max taken as the first logit": ("      if (row[e] > m) m = row[e];", "      (void)m;"),
    "exp with a wrong 1/5! coefficient": ("8.33333333333333333e-3f,", "8.33333333333333333e-2f,"),
    "exp rounds n towards zero": ("const float n = std::rint(x * 1.44269504088896341f);",
                                  "const float n = std::trunc(x * 1.44269504088896341f);"),
    "permute copies the slot's row": ("out[p * H + h] = input[t * H + h];",
                                      "out[p * H + h] = input[(p / K) * H + h];"),
    "one group too many kept": (
        "for (int32_t m = 0; m < topk_group; ++m) {",
        "for (int32_t m = 0; m < topk_group + (topk_group < n_groups ? 1 : 0); ++m) {"),
    "group score from the unbiased scores": (
        "group_vals.assign(b.begin() + j * S, b.begin() + (j + 1) * S);",
        "group_vals.assign(s + j * S, s + (j + 1) * S);"),
    "normalisation sum skips the first weight": (
        "for (int32_t k = 0; k < K; ++k) sum = sum + w[k];",
        "for (int32_t k = 1; k < K; ++k) sum = sum + w[k];"),
    "CSR starts one past": ("expert_start_indices[active] = offset;",
                            "expert_start_indices[active] = offset + 1;"),
    "group limit ignored": (
        "for (int32_t m = 0; m < topk_group; ++m) {", "for (int32_t m = 0; m < n_groups; ++m) {"),
    "experts ranked by the unbiased score": (
        "if (b[x] != b[y]) return b[x] > b[y];\n      return x < y;",
        "if (s[x] != s[y]) return s[x] > s[y];\n      return x < y;"),
    "scaling before the normalisation": (
        "    if (norm_weights) {\n      float sum = 0.0f;\n"
        "      for (int32_t k = 0; k < K; ++k) sum = sum + w[k];\n"
        "      for (int32_t k = 0; k < K; ++k) w[k] = w[k] / sum;\n    }\n"
        "    for (int32_t k = 0; k < K; ++k) w[k] = w[k] * scale;",
        "    for (int32_t k = 0; k < K; ++k) w[k] = w[k] * scale;\n"
        "    if (norm_weights) {\n      float sum = 0.0f;\n"
        "      for (int32_t k = 0; k < K; ++k) sum = sum + w[k];\n"
        "      for (int32_t k = 0; k < K; ++k) w[k] = w[k] / sum;\n    }"),
    "sigmoid of the negated logit": ("out[i] = 1.0f / (1.0f + exp_cody_waite(-x[i]));",
                                     "out[i] = 1.0f / (1.0f + exp_cody_waite(x[i]));"),
    "scale offsets for idle experts too": (
        "    if (count[e] == 0) continue;\n    out[j++] = static_cast<uint32_t>(offset);",
        "    out[j++] = static_cast<uint32_t>(offset);"),
    "scale offsets tail left at zero": (
        "for (; j <= E; ++j) out[j] = static_cast<uint32_t>(offset);",
        "for (; j <= E; ++j) out[j] = 0u;"),
    "stats max taken from the last expert": ("max_count = std::max(max_count, count[e]);",
                                             "max_count = count[e];"),
    "active experts walked in descending id": (
        "for (int32_t e = 0; e < E; ++e) {\n    max_count",
        "for (int32_t e = E - 1; e >= 0; --e) {\n    max_count"),
    "permute ignores token_expert_order": ("const int64_t slot = token_expert_order[p];",
                                           "const int64_t slot = p;"),
    "fp64 finalize drops the weights": ("acc += static_cast<double>(w[t * K + k]) *",
                                        "acc += 1.0 *"),
    "selected-token finalize ignores the selection": (
        "int rc = finalize_one_token(down, restore, w, T, K, H, tokens[j], out + j * H);",
        "int rc = finalize_one_token(down, restore, w, T, K, H, j, out + j * H);"),
    "expert_ids tail padded with 0": ("for (uint32_t j = active; j < static_cast<uint32_t>(E); ++j) "
                                      "expert_ids[j] = -1;",
                                      "for (uint32_t j = active; j < static_cast<uint32_t>(E); ++j) "
                                      "expert_ids[j] = 0;"),
}


def _pins():
    """The oracle's pins, as plain callables (all CPU, a few seconds in total)."""
    return [
        lambda: tr.test_golden_fixtures("route_group_limited.json"),
        lambda: tr.test_golden_fixtures("route_ungrouped_no_norm.json"),
        tr.test_brute_force_tiny_workload,
        lambda: tr.test_brute_force_random(12, 3, 2, 4, True),
        lambda: tr.test_brute_force_random(8, 1, 1, 2, False),
        lambda: tr.test_tie_stress_brute_force("quantised"),
        tr.test_all_equal_scores_pick_lowest_indices,
        tr.test_bias_changes_selection_but_not_weights,
        ti.test_golden_fixture,
        lambda: ti.test_random_ids(1000, 64),
        ti.test_all_slots_on_one_expert,
        tf.test_golden_fixture,
        tf.test_permutation_copy_closed_form,
        lambda: tf.test_library_gather_weighted_sum(33, 8, 256),
        lambda: tf.test_library_gather_weighted_sum(17, 3, 72),
        tf.test_tiny_workload_chain,
        tf.test_fp64_variant_bounds_fp32,
        tf.test_selected_tokens_match_full,
        tp.test_golden_fixture,
        lambda: tp.test_library_gather(64, 4, 24),
        lambda: tp.test_round_trip_through_finalize(2),
        tsc.test_golden_fixture,
        tsg.test_error_bound_on_a_grid,
        tsg.test_special_values,
        lambda: tsm.test_error_bound_against_float64(256),
        tsm.test_large_logits_need_the_max_shift,
        tsm.test_all_equal_row_is_exactly_uniform,
        tsm.test_one_dominant_logit,
        tex.test_binade_endpoints_within_bound,
        tex.test_exact_points_and_clamp,
    ]


def _build_mutant(tmpdir, old, new):
    src = open(ORACLE_SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    path = os.path.join(tmpdir, "mutant.cpp")
    with open(path, "w") as fh:
        fh.write(src.replace(old, new))
    # the copy includes the real header
    inc = os.path.dirname(ORACLE_SRC)
    so = os.path.join(tmpdir, "libmutant.so")
    subprocess.run(["g++", "-O1", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared",
                    "-I", inc, "-o", so, path], check=True)
    return so


def test_pins_pass_on_the_real_oracle():
    for pin in _pins():
        pin()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    old, new = MUTANTS[name]
    with tempfile.TemporaryDirectory() as tmp:
        so = _build_mutant(tmp, old, new)
        caught = []
        with oracle.using_library(so):
            for pin in _pins():
                try:
                    with np.errstate(all="ignore"):
                        pin()
                except (AssertionError, oracle.OracleError, ValueError, IndexError):
                    caught.append(pin)
        assert caught, f"no pin caught the planted mistake: {name}"
