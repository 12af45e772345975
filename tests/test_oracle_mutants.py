"""Plant plausible mistakes in a copy of the oracle and check that the pins in
test_oracle.py catch every one of them (CPU only).

Each mutant is the oracle source with one textual edit, compiled into a
temporary directory; the real oracle is untouched.
"""
import os
import subprocess

import pytest

import oracle as oracle_pkg
from oracle import Oracle, load

import test_oracle as pins
import test_oracle_fp8 as pins8

MUTANTS = {
    "tie_break_to_higher_index": ("l[e] > l[best]", "l[e] >= l[best]"),
    "silu_sign": ("std::exp(-z)", "std::exp(z)"),
    "gate_up_swapped": ("h[i] = (float)(silu(g) * u);", "h[i] = (float)(silu(u) * g);"),
    "down_transposed": ("o += (double)h[i] * (double)wd[i];",
                        "o += (double)h[i] * (double)Wd[i * H + c];"),
    "renorm_inverted": ("if (renorm) {", "if (!renorm) {"),
    "bias_dropped": ("if (bias) s += (double)bias[e];", ";"),
    "gate_weight_dropped": ("acc[c] += (double)w[t * k + r] * o[c];", "acc[c] += o[c];"),
    "shared_dropped": ("      for (int64_t c = 0; c < H; ++c) acc[c] += o[c];\n    }",
                       "    }"),
    "permute_unstable": ("  for (int64_t s = 0; s < T * k; ++s) {\n    const int64_t e = ids[s];",
                         "  for (int64_t s = T * k - 1; s >= 0; --s) {\n    const int64_t e = ids[s];"),
    "logit_index_transposed": ("(double)Wr[e * H + c]", "(double)Wr[c * E + e]"),
    "group_score_is_sum": ("if (l[e] > best) best = l[e];", "best += l[e];"),
    "group_tie_break_to_higher_index": ("score[j] > score[bj]", "score[j] >= score[bj]"),
    "group_mask_ignored": ("if (taken[e] || !kept[e / G]) continue;", "if (taken[e]) continue;"),
    "e4m3_ties_away_from_zero": ("if (rem > 0.5 || (rem == 0.5 && std::fmod(n, 2.0) != 0.0)) n += 1.0;",
                                 "if (rem >= 0.5) n += 1.0;"),
    "e4m3_row_scale_one_too_small": ("e = (2.0 * f <= 1.75) ? E - 8 : E - 7;", "e = E - 8;"),
    "e4m3_exponent_bias": ("ef == 0 ? std::ldexp((double)m / 8.0, -6)\n                             : std::ldexp(1.0 + (double)m / 8.0, ef - 7);",
                           "ef == 0 ? std::ldexp((double)m / 8.0, -6)\n                             : std::ldexp(1.0 + (double)m / 8.0, ef - 8);"),
}

PIN_CALLS = [
    lambda o: pins.test_logits_match_float64_matmul(o),
    lambda o: pins.test_topk_ids_match_stable_sort(o, 40, 7),
    lambda o: pins.test_topk_all_equal_logits(o),
    lambda o: pins.test_topk_k_equals_E_is_permutation(o),
    lambda o: pins.test_weights_renorm_sum_to_one_and_match_softmax(o),
    lambda o: pins.test_weights_no_renorm_is_full_softmax(o),
    lambda o: pins.test_weights_k1_is_exactly_one(o),
    lambda o: pins.test_permute_is_stable_counting_sort(o, 100, 16, 4, 1),
    lambda o: pins.test_dense_bruteforce_equals_sparse(o),
    lambda o: pins.test_k_equals_E_uniform_is_mean_of_experts(o),
    lambda o: pins.test_single_expert_is_dense_swiglu_in_torch_float64(o),
    lambda o: pins.test_shared_expert_adds_dense_ffn(o),
    lambda o: pins.test_token_permutation_equivariance(o),
    lambda o: pins.test_stages_compose_to_forward(o),
    lambda o: pins.test_closed_form_golden(o),
    lambda o: pins.test_grouped_topk_matches_bruteforce(o, 16, 3, 4, 2),
    lambda o: pins.test_grouped_topk_matches_bruteforce(o, 64, 8, 8, 3),
    lambda o: pins.test_grouped_topk_reduces_to_plain_topk(o),
    lambda o: pins.test_grouped_topk_stays_in_kept_groups(o),
    lambda o: pins8.test_decode_every_code_matches_torch(o),
    lambda o: pins8.test_encode_round_trips_and_rounds_ties_to_even(o),
    lambda o: pins8.test_encode_random_values_match_torch(o, 0),
    lambda o: pins8.test_quantize_rows_follow_the_rule(o),
]


def _failures(orc):
    n = 0
    for call in PIN_CALLS:
        try:
            call(orc)
        except AssertionError:
            n += 1
    return n


def test_unmutated_oracle_passes_every_pin():
    assert _failures(Oracle()) == 0


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    src = open(oracle_pkg._SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new)
    cpp = tmp_path / "mutant.cpp"
    cpp.write_text(mutated)
    so = tmp_path / "libmutant.so"
    subprocess.run(["g++", "-std=c++17", "-O1", "-fopenmp", "-fPIC", "-shared",
                    "-ffp-contract=off", str(cpp), "-o", str(so)], check=True)
    orc = Oracle(load(str(so)))
    assert _failures(orc) >= 1, f"no pin caught the planted mistake {name}"
