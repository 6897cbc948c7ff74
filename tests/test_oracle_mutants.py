"""The oracle's pins are strong enough to catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (on the CPU,
in a temporary directory), compiles it, and runs the pins that should catch it
against the mutant: at least one of them must fail. The committed oracle is
never modified.
"""
import os

import numpy as np
import pytest

import oracle
import test_oracle_attention as TA
import test_oracle_formats as TF
import test_oracle_prepare as TP

MUTANTS = [
    # (name, original text, mistaken text, pins that should catch it)
    ("rope_sign_swapped", "(c % 2 == 0) ? a - b : a + b", "(c % 2 == 0) ? a + b : a - b",
     [TP.test_rope_is_the_complex_rotation]),
    ("rope_partner_dropped", "float p = y[c ^ 1]", "float p = y[c]",
     [TP.test_rope_is_the_complex_rotation]),
    ("rope_frequency_index", "co = cs[c / 2], si = sn[c / 2]", "co = cs[c % 32], si = sn[c % 32]",
     [TP.test_rope_is_the_complex_rotation]),
    ("rms_mean_dropped", "sqrt(sumsq / ORC_D + (double)eps)", "sqrt(sumsq + (double)eps)",
     [TP.test_rmsnorm_unit_rms_and_zero_head]),
    ("k_head_offset", "(h - hq)) * ORC_D + c] = orc_e4m3_code((double)key)",
     "(h - hq - hkv + 1)) * ORC_D + c] = orc_e4m3_code((double)key)",
     [lambda: TP.test_columns_feed_only_their_head("k1", (TP.KCOL + 64, TP.KCOL + 128), "k1")]),
    ("round_truncates", "return rint(v / q) * q;", "return trunc(v / q) * q;",
     [TF.test_e4m3_encode_matches_torch_in_range, TF.test_bf16_matches_torch]),
    ("ties_away_from_zero", "return rint(v / q) * q;", "return round(v / q) * q;",
     [TF.test_e4m3_round_trip_and_saturation, TF.test_bf16_matches_torch]),
    ("window_off_by_one", "p - cfg->window + 1 > 0 ? p - cfg->window + 1 : 0",
     "p - cfg->window > 0 ? p - cfg->window : 0",
     [TA.test_window_keeps_token_and_2047_before_it]),
    ("causal_sees_next_token", "const int64_t p = n - ql + i;",
     "const int64_t p = (i + 1 < ql) ? n - ql + i + 1 : n - ql + i;",
     [TA.test_verify_block_is_causal]),
    ("gqa_head_map", "const int g = h / group;", "const int g = h % hkv;",
     [lambda: TA.test_matches_dense_brute_force(1, 1, 0, (5, 11), 1.0)]),
    ("softmax_scale_dropped", "s[j - lo] = dot * scale;", "s[j - lo] = dot;",
     [lambda: TA.test_matches_dense_brute_force(1, 1, 0, (5, 11), 1.0)]),
    ("v_scale_dropped", "ORC_D + c]] * vs);", "ORC_D + c]]);",
     [lambda: TA.test_matches_dense_brute_force(8, 4, 5, (0, 13), 0.5)]),
    ("page_offset_transposed", "r = page * P + j % P;", "r = page * P + (j / P) % P;",
     [lambda: TA.test_matches_dense_brute_force(1, 4, 3, (6, 16), 0.5)]),
    ("sigmoid_sign", "1.0 / (1.0 + exp(-g))", "1.0 / (1.0 + exp(g))",
     [TA.test_normgate_saturated_gate_is_plain_rmsnorm]),
    # (mistakes that stay inside the arrays: a mutant runs in the test's process)
    ("ragged_rows_reversed", "const int64_t t = cu_seqlens_q[b] + i;",
     "const int64_t t = cu_seqlens_q[b + 1] - 1 - i;",
     [lambda: TA.test_ragged_batch_matches_dense_brute_force(0)]),
    # the scaled cache path ("012-attention-local-splits.py", `_prepare_qkv`, `if SCALED:`)
    ("k_divided_by_v_scale", "(key / k_scale)", "(key / v_scale)",
     [TP.test_scaled_cache_codes_from_the_definition]),
    ("v_divided_by_k_scale", "(value / v_scale)", "(value / k_scale)",
     [TP.test_scaled_cache_codes_from_the_definition]),
    ("no_bf16_after_k_scale", "key = (float)orc_bf16_round((double)(key / k_scale));", "key = key / k_scale;",
     [TP.test_scaled_cache_codes_from_the_definition]),
    # q_norm 1 (the vLLM CuTeDSL qk_norm page, QKNormDirectKernel.kernel: float32
    # through the scale, the store the only rounding)
    ("q_norm_bf16_before_scale", "const float scaled_q = normed * cfg->qk_scale_factor;",
     "const float scaled_q = (float)orc_bf16_round((double)normed) * cfg->qk_scale_factor;",
     [TP.test_folded_q_norm_is_one_bf16_rounding_of_the_float32_chain]),
    ("q_norm_scale_dropped", "const float scaled_q = normed * cfg->qk_scale_factor;",
     "const float scaled_q = normed;",
     [TP.test_folded_q_norm_is_one_bf16_rounding_of_the_float32_chain]),
    ("q_norm_factor_kept_in_softmax", "cfg->q_norm == 1 ? (double)cfg->sm_scale",
     "cfg->q_norm == 1 ? (double)(float)((double)cfg->sm_scale * (double)cfg->qk_scale_factor)",
     [TA.test_folded_q_norm_matches_dense_brute_force]),
    ("no_bf16_after_v_scale", "value = (float)orc_bf16_round((double)(value / v_scale));",
     "value = value / v_scale;", [TP.test_scaled_cache_codes_from_the_definition]),
]


@pytest.mark.parametrize("name,orig,bad,pins", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, orig, bad, pins, tmp_path):
    src = oracle.source()
    assert src.count(orig) >= 1, f"mutation site not found: {orig}"
    lib = oracle.compile_source(src.replace(orig, bad), os.path.join(tmp_path, f"mut_{name}.so"))
    caught = []
    with oracle.use_library(lib):
        for pin in pins:
            try:
                pin()
            except AssertionError:
                caught.append(pin)
    assert caught, f"no pin caught the planted mistake {name}"
    # and the real oracle still passes the same pins
    for pin in pins:
        pin()
