"""Planted mistakes in the oracle must fail a pin.

Each case copies moe_oracle.c, plants one plausible mistake (a dropped term, a
wrong index, a flipped comparison, a floor for a ceiling ...), builds it, and
checks that at least one of the pins in test_oracle_pins.py fails against it.
The real oracle source is never modified.
"""
from __future__ import annotations

import os
import subprocess
import tempfile

import pytest

import oracle
from oracle import build as obuild
from tests import test_oracle_pins as pins

MUTATIONS = {
    "butterfly_drops_partner": ("t[p] = s[p] + s[p ^ o];", "t[p] = s[p] + s[p];"),
    "lane_layout_interleaved": ("int h = stripe + 8 * p + t;", "int h = stripe + p + 32 * t;"),
    "stripe_order_reversed": ("for (int stripe = 0; stripe < H; stripe += 256)",
                              "for (int stripe = H - 256; stripe >= 0; stripe -= 256)"),
    "ties_to_higher_id": ("if (best < 0 || key > bk)", "if (best < 0 || key >= bk)"),
    "exp_drops_ln2_tail": ("r = fmaf(-n, LN2_LO, r);", "r = r;"),
    "exp_short_taylor": ("float p = C[7];", "float p = 0.0f;"),
    "weights_not_normalised": ("w[j] = a[j] / S;", "w[j] = a[j];"),
    "coreset_ascending_mass": ("Q[order[p]] < Q[e]", "Q[order[p]] > Q[e]"),
    "threshold_floor": ("if ((q << s) != prod) q += 1;", ";"),
    "threshold_strict": ("while (c < cap && run < theta)", "while (c < cap && run <= theta)"),
    "budget_off_by_one": ("? max_experts : nt;", "? max_experts + 1 : nt;"),
    "budget_ignored_without_tau": ("const int renorm = tau < 1.0f || cap < nt;",
                                   "const int renorm = tau < 1.0f;"),
    "renorm_over_all_slots": ("if (idx[j] >= 0 && idx[j] < E && in_core[idx[j]]) s = s + w[j];",
                              "s = s + w[j];"),
    "disabled_redivides": ("for (int j = 0; j < k; ++j) wo[j] = w[j];\n                continue;",
                           "for (int j = 0; j < k; ++j) wo[j] = w[j];"),
    "silu_sign": ("hbuf[i] = g / (1.0 + exp(-g)) * u;", "hbuf[i] = g / (1.0 + exp(g)) * u;"),
    "forward_first_slot_weight": ("double wj = (double)J->w_renorm[(size_t)r * J->k + j];",
                                  "double wj = (double)J->w_renorm[(size_t)r * J->k];"),
    "forward_drops_shared": ("moe_oracle_expert_ffn(xr, J->sg, J->su, J->sd, J->H, J->Is, yr);",
                             "memset(yr, 0, sizeof(double) * (size_t)J->H);"),
    "down_proj_transposed": ("const uint16_t* dh = wd + (size_t)h * I;",
                             "const uint16_t* dh = wd + (size_t)(h % I) * I;"),
    "weight_sum_in_id_order": (
        "            S = S + a[j];\n        }",
        "        }\n        for (int e = 0; e < J->E; ++e)\n"
        "            for (int j = 0; j < J->k; ++j)\n"
        "                if (idx[j] == e) S = S + a[j];"),
    "prob_denominator_in_id_order": (
        "for (int e = p; e < J->E; e += 32) acc = acc + moe_oracle_exp_c(z[e] - m);",
        "if (p == 0) for (int e = 0; e < J->E; ++e) acc = acc + moe_oracle_exp_c(z[e] - m);"),
    "prob_denominator_drops_butterfly": ("for (int p = 0; p < 32; ++p) t[p] = d[p] + d[p ^ o];",
                                         "for (int p = 0; p < 32; ++p) t[p] = d[p];"),
    "prob_mass_ignored": ("float wj = (topk_mass ? topk_mass : topk_w)[(size_t)r * k + j];",
                          "float wj = topk_w[(size_t)r * k + j];"),
    "dequant_nibble_order": ("int nib = (k & 1) ? (byte >> 4) : (byte & 0xF);",
                             "int nib = (k & 1) ? (byte & 0xF) : (byte >> 4);"),
    "dequant_nibble_unsigned": ("qv = nib >= 8 ? nib - 16 : nib;", "qv = nib;"),
    "dequant_scales_row_major": ("d[(size_t)(k / 32) * rows + r]", "d[(size_t)r * (K / 32) + k / 32]"),
    "dequant_truncates": ("return (uint16_t)((u + 0x7FFFu + lsb) >> 16);",
                          "return (uint16_t)(u >> 16);"),
}

PINS = [
    pins.test_exp_c_special_values, pins.test_exp_c_within_two_ulp_of_exp,
    pins.test_logit_lane_order_hand_value, pins.test_logit_butterfly_hand_value,
    pins.test_logit_stripe_order_hand_value, pins.test_logit_within_summation_bound,
    pins.test_topk_is_sorted_selection, pins.test_topk_ties_go_to_lower_id,
    pins.test_weights_equal_full_softmax_then_renormalised,
    pins.test_coreset_brute_force_tiny_config, pins.test_coreset_threshold_hand_example,
    pins.test_coreset_threshold_is_ceiling, pins.test_coreset_disabled_is_plain_topk,
    pins.test_expert_ffn_hand_value, pins.test_expert_ffn_matches_dense_fp64,
    pins.test_forward_matches_dense_moe_fp64,
    pins.test_coreset_budget_hand_example,
    pins.test_weight_sum_in_rank_order_hand_case,
    pins.test_prob_mass_denominator_in_lane_order_hand_case,
    pins.test_prob_mass_equals_full_softmax, pins.test_coreset_prob_mass_changes_membership,
    pins.test_dequant_hand_cases,
] + [lambda m, s=s: pins.test_coreset_prob_mass_brute_force_random_tiny(m, s) for s in range(2)] \
  + [lambda m, s=s: pins.test_coreset_brute_force_random_tiny(m, s) for s in range(4)] \
  + [lambda m, s=s: pins.test_coreset_budget_brute_force_random_tiny(m, s) for s in range(4)]


def _build_mutant(name: str, tmp: str) -> str:
    old, new = MUTATIONS[name]
    src = open(obuild.SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique/found: {name}"
    path = os.path.join(tmp, f"{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    so = os.path.join(tmp, f"lib{name}.so")
    subprocess.run(["gcc", *obuild.CFLAGS, "-w", path, "-o", so, "-lm", "-lpthread"], check=True)
    return so


def _fails_some_pin() -> bool:
    for pin in PINS:
        try:
            pin(oracle)
        except Exception:
            return True
    return False


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name):
    with tempfile.TemporaryDirectory() as tmp:
        so = _build_mutant(name, tmp)
        try:
            oracle.use_library(so)
            assert _fails_some_pin(), f"no pin caught the planted mistake {name!r}"
        finally:
            oracle.use_library(None)


def test_unmutated_oracle_passes_every_pin():
    oracle.use_library(None)
    assert not _fails_some_pin()
