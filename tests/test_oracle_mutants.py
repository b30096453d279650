"""The oracle's pins must catch plausible mistakes.

Each case copies ``oracle/msa_oracle.c``, plants one mistake in the copy (on
the CPU, in a temporary directory), compiles it and runs the pins from
``test_oracle_pins`` against it: at least one pin has to fail.  The real oracle
is restored afterwards.
"""
import os
import shutil
import subprocess

import pytest

import oracle
import test_oracle_fp8_index_pins as fp8_index_pins
import test_oracle_fp8_pins as fp8_pins
import test_oracle_pins as pins
import test_oracle_prologue_pins as prologue_pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "msa_oracle.c")

MUTANTS = {
    "pool_ignores_causality": ("const int j_end = ((b + 1) * block < pos + 1) ? (b + 1) * block : pos + 1;",
                               "const int j_end = ((b + 1) * block < kv_len) ? (b + 1) * block : kv_len;"),
    "ties_go_to_higher_index": ("pooled_row[b] > pooled_row[best]) best = b;",
                                "pooled_row[b] >= pooled_row[best]) best = b;"),
    "local_block_not_forced": ("if (k > 0) taken[local] = 1;", ""),
    "attention_ignores_causality": ("j <= pos; ++j) key[n++] = j;", "1; ++j) key[n++] = j;"),
    "scale_dropped": ("x[t] = scale * acc;", "x[t] = acc;"),
    "wrong_group_of_head": ("const int g = h / G;", "const int g = h % hkv;"),
    "top_left_alignment": ("const int pos = kv_len - q_len + (i - cu_q[s]);",
                           "const int pos = (i - cu_q[s]);"),
    "lse_without_max": ("lse[(size_t)r * hq + h] = m + log(l);", "lse[(size_t)r * hq + h] = log(l);"),
    "index_dot_skips_last_dim": ("for (int d = 0; d < n; ++d)", "for (int d = 0; d + 1 < n; ++d)"),
    "value_from_wrong_row": ("const uint16_t *vj = v + ((size_t)(cu_k[s] + key[t]) * hkv + g)",
                             "const uint16_t *vj = v + ((size_t)(key[t]) * hkv + g)"),
    # fp8 K/V
    "e4m3_exponent_bias_8": ("ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)"),
    "e4m3_ties_round_up": ("else pick = (c % 2 == 0) ? c : c + 1;", "else pick = c + 1;"),
    "e4m3_no_saturation": ("if (a >= 448.0) return (uint8_t)(sign | 0x7E);", "if (a >= 448.0) return 0x7F;"),
    "fp8_scale_for_max_240": ("amax > 0.f ? amax / 448.0f : 1.0f", "amax > 0.f ? amax / 240.0f : 1.0f"),
    "fp8_scale_row_ignores_sequence": ("k_scale[(size_t)(blk0[s] + key[t] / block) * hkv + g]",
                                       "k_scale[(size_t)(key[t] / block) * hkv + g]"),
    "fp8_value_scale_dropped": ("oh[d] += p * (msa_oracle_e4m3_value(vj[d]) * sv);",
                                "oh[d] += p * msa_oracle_e4m3_value(vj[d]);"),
    # fp8 index
    "fp8_index_key_scale_row_ignores_sequence": ("(double)in->k_scale[blk0 + j / block]",
                                                 "(double)in->k_scale[j / block]"),
    "fp8_index_query_scale_of_group_0": ("(double)in->q_scale[(size_t)i * hkv + g]",
                                         "(double)in->q_scale[(size_t)i * hkv]"),
    "fp8_index_key_scale_dropped": ("msa_oracle_e4m3_value(in->k8[e]) * (double)in->k_scale[blk0 + j / block]",
                                    "msa_oracle_e4m3_value(in->k8[e])"),
    # index prologue
    "rope_rotation_sign": ("out[j] = y[j] * c - y[j + half] * sn;", "out[j] = y[j] * c + y[j + half] * sn;"),
    "rope_frequency_exponent": ("pow(rope_base, -2.0 * j / rope_dim)", "pow(rope_base, -1.0 * j / rope_dim)"),
    "rms_norm_sum_not_mean": ("sqrt(ss / d_idx + eps)", "sqrt(ss + eps)"),
    "norm_weight_dropped": ("y[d] = y[d] * inv * bf16_bits_to_double(gamma[d]);", "y[d] = y[d] * inv;"),
    "key_head_takes_query_norm_weight": ("(h < hkv) ? gamma_q : gamma_k", "gamma_q"),
}

PIN_TESTS = [
    lambda: pins.test_golden_three_block_example(),
    lambda: pins.test_pooled_matches_torch_matmul(0),
    lambda: pins.test_select_matches_full_sort_with_ties(0),
    lambda: pins.test_attention_matches_masked_sdpa(0),
    lambda: pins.test_forward_equals_dense_causal_when_k_covers_all_blocks(),
    lambda: pins.test_invariants_on_tiny_workload(),
    lambda: pins.test_token_budget_and_closed_forms(),
    lambda: fp8_pins.test_e4m3_golden_table(),
    lambda: fp8_pins.test_e4m3_values_match_torch_for_every_code(),
    lambda: fp8_pins.test_e4m3_codes_match_torch_rounding(),
    lambda: fp8_pins.test_quantizer_scale_and_error_bound(),
    lambda: fp8_pins.test_attention_fp8_equals_bf16_attention_on_the_fp8_grid(),
    lambda: fp8_index_pins.test_pooled_fp8_equals_bf16_pooled_on_the_fp8_grid(),
    lambda: fp8_index_pins.test_pooled_fp8_matches_brute_force_with_quantizer_scales(),
    lambda: fp8_index_pins.test_index_fp8_is_the_selection_over_pooled_fp8(),
    lambda: fp8_index_pins.test_quantize_index_fp8_scales_and_extremes(),
    lambda: prologue_pins.test_identity_projection_matches_torch_rms_norm(),
    lambda: prologue_pins.test_rms_norm_is_scale_invariant_and_normalises_constants(),
    lambda: prologue_pins.test_rope_is_a_complex_rotation_of_each_pair(4, 100.0),
    lambda: prologue_pins.test_rope_position_zero_is_identity_and_dots_depend_on_offsets_only(),
]


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = text.replace(old, new)
    src = tmp_path / "mutant.c"
    src.write_text(mutated)
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-fopenmp", "-shared", "-o", str(lib), str(src),
                    "-lm"], check=True)
    failures = 0
    oracle.use_library(str(lib))
    try:
        for t in PIN_TESTS:
            try:
                t()
            except (AssertionError, ValueError):
                failures += 1
    finally:
        oracle.use_library(None)
    assert failures > 0, f"no pin caught the mutant {name}"
