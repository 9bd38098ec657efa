"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check that
the pins in test_oracle_pins.py, test_oracle_fp8.py, test_oracle_w8a8.py,
test_oracle_a2.py and test_oracle_blocks.py catch every one of them."""
import ctypes
import os

import pytest

import oracle
from tests import test_oracle_fp8 as pins8
from tests import test_oracle_pins as pins
from tests import test_oracle_a2 as pins_a2
from tests import test_oracle_blocks as pins_blk
from tests import test_oracle_w8a8 as pins_a8

SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.c")

# (name, exact text in moe_oracle.c, replacement)
MUTATIONS = [
    ("ties_to_higher_index", "if (best < 0 || key[e] > key[best])", "if (best < 0 || key[e] >= key[best])"),
    ("softmax_sign", "w[j] = exp(key[idx[j]] - kmax);", "w[j] = exp(kmax - key[idx[j]]);"),
    ("silu_sign", "double silu = g / (1.0 + exp(-g));", "double silu = g / (1.0 + exp(g));"),
    ("dropped_up_projection", "h[i] = silu * u;", "h[i] = silu;"),
    ("transposed_down_projection", "load_weight(w_down, wd_off + j * I + i) * h[i]",
     "load_weight(w_down, wd_off + i * d + j) * h[i]"),
    ("swapped_gate_and_up", "double silu = g / (1.0 + exp(-g));\n        h[i] = silu * u;",
     "double silu = u / (1.0 + exp(-u));\n        h[i] = silu * g;"),
    ("dropped_bias", "const double b = bias ? bias[e] : 0.0;", "const double b = 0.0;"),
    ("dropped_shared_in_combine", "double acc = y_shared ? y_shared[t * d + c] : 0.0;",
     "double acc = 0.0;"),
    ("first_weight_for_all_slots", "acc += topk_w[t * K + j] * y_perm[p * d + c];",
     "acc += topk_w[t * K] * y_perm[p * d + c];"),
    ("reversed_order_within_expert", "int32_t p = cursor[topk_idx[f]]++;",
     "int32_t p = offsets[topk_idx[f] + 1] - 1 - (cursor[topk_idx[f]]++ - offsets[topk_idx[f]]);"),
    ("sigmoid_sign", "aff[e] = 1.0 / (1.0 + exp(-s[e]));", "aff[e] = 1.0 / (1.0 + exp(s[e]));"),
    ("bias_leaks_into_sigmoid_weights", "w[j] = aff[idx[j]] / (denom + 1e-6);",
     "w[j] = key[idx[j]] / (denom + 1e-6);"),
    ("router_reads_wrong_row", "load_elem(w_g, dtype, e * d + k)", "load_elem(w_g, dtype, ((e + 1) % E) * d + k)"),
    ("e4m3_exponent_bias", "v = ldexp(8.0 + M, E - 10);", "v = ldexp(8.0 + M, E - 11);"),
    ("e4m3_subnormal_step", "v = ldexp((double)M, -9);", "v = ldexp((double)M, -10);"),
    ("e4m3_round_half_up", "nearbyint(a / unit)", "floor(a / unit + 0.5)"),
    ("e4m3_no_saturation", "return sgn | 0x7E;", "return sgn | 0x7F;"),
    ("fp8_scale_by_column", "sc = (double)w->scale[r];", "sc = (double)w->scale[i % w->row_len];"),
    ("fp8_down_scale_row_length", "fp8_weight(w_down, s_down, I), fp8_weight(ws_gate",
     "fp8_weight(w_down, s_down, d), fp8_weight(ws_gate"),
    ("quant_scale_not_amax", "amax / 448.0f : 1.0f;\n    for (int64_t c = 0; c < n; ++c)\n        codes[c]",
     "amax / 240.0f : 1.0f;\n    for (int64_t c = 0; c < n; ++c)\n        codes[c]"),
    ("a2_scale_not_amax", "amax / 448.0f : 1.0f;\n    for (int64_t c = 0; c < n; ++c) {\n        const float q",
     "amax / 240.0f : 1.0f;\n    for (int64_t c = 0; c < n; ++c) {\n        const float q"),
    ("a8_x_not_quantised", "act_hat(s, d, planes, s->xh);",
     "for (int64_t k = 0; k < d; ++k) s->xh[k] = (double)s->f[k];"),
    ("a8_h_not_rounded_to_bf16", "s->f[i] = round_bf16((float)s->h[i]);",
     "s->f[i] = (float)s->h[i];"),
    ("a8_h_not_quantised", "act_hat(s, I, planes, s->h);",
     "for (int64_t i = 0; i < I; ++i) s->h[i] = (double)s->f[i];"),
    ("a8_h_read_as_two_planes", "act_hat(s, I, planes, s->h);", "act_hat(s, I, 2, s->h);"),
    ("a8_bf16_rounds_half_up", "u += 0x7fffu + ((u >> 16) & 1u);", "u += 0x8000u;"),
    ("a8_down_scale_row_length", "fp8w(w_down, s_down, I, blocks), y_perm,",
     "fp8w(w_down, s_down, d, blocks), y_perm,"),
    ("a8_shared_expert_skipped", "swiglu_row_a8(d, c->Is, c->dtype, c->x, t * d, &c->ws_gate",
     "if (0) swiglu_row_a8(d, c->Is, c->dtype, c->x, t * d, &c->ws_gate"),
    ("a2_lo_plane_dropped",
     "out[k] = (e4m3_value(s->c[k]) + e4m3_value(s->c2[k])) * (double)sc;",
     "out[k] = e4m3_value(s->c[k]) * (double)sc;"),
    ("a2_remainder_of_the_unscaled_value", "const float r = q - (float)e4m3_value(hi[c]);",
     "const float r = v[c] - (float)e4m3_value(hi[c]);"),
    ("a2_remainder_plane_scaled_twice",
     "out[k] = (e4m3_value(s->c[k]) + e4m3_value(s->c2[k])) * (double)sc;",
     "out[k] = (e4m3_value(s->c[k]) + e4m3_value(s->c2[k]) * (double)sc) * (double)sc;"),
    ("a2_one_plane_in_the_token_layer",
     "logits, nthreads, 2,\n                             0);",
     "logits, nthreads, 1,\n                             0);"),
    ("block_scale_ignores_the_column_block",
     "sc = (double)w->scale[(r / w->block) * nbc + c / w->block];",
     "sc = (double)w->scale[(r / w->block) * nbc];"),
    ("block_scale_ignores_the_row_block",
     "sc = (double)w->scale[(r / w->block) * nbc + c / w->block];",
     "sc = (double)w->scale[c / w->block];"),
    ("block_down_row_length",
     "fp8_block_weight(w_down, s_down, I),\n                             fp8_block_weight(ws_gate",
     "fp8_block_weight(w_down, s_down, d),\n                             fp8_block_weight(ws_gate"),
    ("block_stage_down_row_length", "fp8_block_weight(w_down, s_down, I),\n                      y_perm",
     "fp8_block_weight(w_down, s_down, d),\n                      y_perm"),
    ("block_quant_amax_of_the_first_row", "scale[br * nbc + bc] = quantize_vec(blk, nr * nc, cb);",
     "scale[br * nbc + bc] = quantize_vec(blk, nc, cb);"),
    ("block_quant_codes_transposed", "codes[(r0 + i) * cols + c0 + j] = cb[i * nc + j];",
     "codes[(r0 + i) * cols + c0 + j] = cb[j * nr + i];"),
    ("block_w8a8_stage_with_two_planes",
     "s_down, y_perm, h_pre, h_hat, nthreads, 1, 1);",
     "s_down, y_perm, h_pre, h_hat, nthreads, 2, 1);"),
    ("block_a2_stage_with_one_plane",
     "s_down, y_perm, h_pre, h_hat, nthreads, 2, 1);",
     "s_down, y_perm, h_pre, h_hat, nthreads, 1, 1);"),
]

PIN_TESTS = [
    lambda: pins.test_topk_matches_exhaustive_sort(40, 256, 8, 2),
    lambda: pins.test_ties_go_to_lower_index_and_signed_zero_is_a_tie(),
    lambda: pins.test_K_equals_E_is_full_softmax(),
    lambda: pins.test_weights_sum_to_one(),
    lambda: pins.test_scores_are_x_times_wg_transposed(),
    lambda: pins.test_bias_enters_selection_and_weights(),
    lambda: pins.test_forward_matches_dense_masked_evaluation("f32", 9, 24, 6, 3, 40, 16),
    lambda: pins.test_single_expert_is_a_dense_swiglu_mlp(),
    lambda: pins.test_hand_built_layer_closed_form(),
    lambda: pins.test_combine_is_linear_in_the_weights(),
    lambda: pins.test_permutation_is_the_stable_expert_order(37, 3, 3),
    lambda: pins.test_sigmoid_router_matches_brute_force(40, 64, 6, 4),
    lambda: pins.test_sigmoid_bias_steers_selection_but_not_weights(),
    lambda: pins.test_sigmoid_forward_matches_dense_masked_evaluation("f32"),
    lambda: pins8.test_decode_matches_torch_float8_for_every_code(),
    lambda: pins8.test_encode_is_the_nearest_code_with_ties_to_even(),
    lambda: pins8.test_encode_saturates_and_keeps_nan(),
    lambda: pins8.test_quantised_rows_meet_the_format_error_bound("f32"),
    lambda: pins8.test_fp8_layer_equals_the_layer_on_dequantised_weights("bf16", 0),
    lambda: pins_a8.test_bf16_rounding_matches_torch_including_ties(),
    lambda: pins_a8.test_w8a8_expert_matches_library_quantisation_at_every_step(1, [3, 0, 5, 1]),
    lambda: pins_a8.test_w8a8_layer_equals_the_8bit_weight_layer_when_activations_are_exact(
        "softmax", 32),
    lambda: pins_a2.test_planes_match_torch_float8_casts(),
    lambda: pins_a2.test_planes_meet_the_two_step_error_bound_and_are_not_one_plane(),
    lambda: pins_a2.test_a2_expert_matches_library_casts_at_every_step(1, [3, 0, 5, 1]),
    lambda: pins_a2.test_a2_token_forward_matches_the_expert_stage(),
    lambda: pins_blk.test_block_codes_and_scales_match_torch("f32", (300, 200)),
    lambda: pins_blk.test_block_layer_equals_the_layer_on_dequantised_weights("bf16", 0, 192, 320, 64),
    lambda: pins_blk.test_a2_blocks_expert_matches_library_casts_at_every_step(2, [7, 2]),
    lambda: pins_blk.test_w8a8_blocks_expert_matches_library_quantisation_at_every_step(4, [7, 2]),
    lambda: pins_blk.test_w8a8_blocks_token_forward_matches_the_expert_stage(),
]


def _caught(lib) -> bool:
    saved = oracle._lib
    oracle._lib = lib
    try:
        for t in PIN_TESTS:
            try:
                t()
            except (AssertionError, ValueError):
                return True
        return False
    finally:
        oracle._lib = saved


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique/absent"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    so = oracle.compile_c(str(mutated), str(tmp_path / "libmutant.so"))
    lib = oracle.bind(ctypes.CDLL(so))
    assert _caught(lib), f"no pin caught the planted mistake '{name}'"


def test_unmutated_oracle_passes_every_pin():
    assert not _caught(oracle._load())
