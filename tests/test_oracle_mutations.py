"""The pins must catch plausible mistakes in the oracle (CPU only).

Each case plants one mistake in a temporary copy of oracle/kvq_oracle.c (or
oracle/attention.py),
rebuilds that copy, and runs the pin test expected to catch it against the
copy in a subprocess: that test must fail. The real oracle is not touched.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, original text, planted mistake, pin test that must fail)
MUTANTS = [
    ("ties_all_strict", "int passed = upper_is_even ? (a >= midpoint) : (a > midpoint);",
     "int passed = (a > midpoint);", "test_oracle_pins_formats.py::test_e2m1_midpoints_golden"),
    ("ties_flipped", "int upper_is_even = ((k + 1) % 2) == 0;",
     "int upper_is_even = ((k + 1) % 2) == 1;",
     "test_oracle_pins_formats.py::test_e2m1_midpoints_golden"),
    ("sign_from_signbit", "uint8_t sign = (normalized < 0.0f) ? 8u : 0u;",
     "uint8_t sign = signbit(normalized) ? 8u : 0u;",
     "test_oracle_pins_formats.py::test_e2m1_special_inputs"),
    ("nibbles_swapped", "row[(g0 + j) / 2] = (uint8_t)(lo | (uint8_t)(hi << 4));",
     "row[(g0 + j) / 2] = (uint8_t)(hi | (uint8_t)(lo << 4));",
     "test_oracle_pins_store.py::test_store_low_nibble_holds_lower_index"),
    ("ceil_off_by_one", "if (fraction != 0u) e += 1;", "if (fraction != 0u) e += 0;",
     "test_oracle_pins_formats.py::test_ceil_pow2_exponent_is_exact_ceil_log2"),
    ("zero_group_byte_0", "if (amax == 0.0f) return 0;", "if (amax == 0.0f) return -127;",
     "test_oracle_pins_formats.py::test_mxfp4_zero_group_scale_is_127"),
    ("scale_divisor_4", "float v = amax / 6.0f;", "float v = amax / 4.0f;",
     "test_oracle_pins_formats.py::test_mxfp4_scale_power_of_two_times_six_lands_on_six"),
    ("rope_sign", "float r_even = ec - os;", "float r_even = ec + os;",
     "test_oracle_pins_rope.py::test_quarter_and_half_turns"),
    ("rope_sin_column", "s = cs[32 + (i - 224)];", "s = cs[31 + (i - 224)];",
     "test_oracle_pins_rope.py::test_quarter_and_half_turns"),
    ("table_row_unrounded", "int64_t table_row = (position / compress_ratio) * compress_ratio;",
     "int64_t table_row = position;",
     "test_oracle_pins_rope.py::test_slot_and_ratio_gates_and_table_row"),
    ("ratio_gate", "if ((position + 1) % compress_ratio != 0) return -1;",
     "if (position % compress_ratio != 0) return -1;",
     "test_oracle_pins_rope.py::test_slot_and_ratio_gates_and_table_row"),
    ("mxfp8_cap_ignores_sanitize", "int32_t cap = sanitize ? 254 : 255;", "int32_t cap = 255;",
     "test_oracle_pins_rope.py::test_mxfp8_scale_cap_depends_on_sanitising"),
    ("mxfp8_amax_floor", "const float kMinAmax = 1e-4f;", "const float kMinAmax = 1e-5f;",
     "test_oracle_pins_rope.py::test_worked_records"),
    ("nvfp4_reciprocal", "uint8_t lo = oracle_e2m1_code(x[j] / s);",
     "uint8_t lo = oracle_e2m1_code(x[j] * (1.0f / s));",
     "test_oracle_pins_rope.py::test_nvfp4_division_ties"),
    ("nvfp4_scale_floor", "const float kMinScale = 0.001953125f; /* 2**-9 */",
     "const float kMinScale = 0.015625f;", "test_oracle_pins_rope.py::test_worked_records"),
    ("e4m3_ties_up", "    return (fmodf(lower, 2.0f) == 0.0f) ? lower : lower + 1.0f;",
     "    return lower + 1.0f;", "test_oracle_pins_formats.py::test_e4m3_named_values"),
    ("rmsnorm_eps_dropped", "float var = mean + eps;", "float var = mean;",
     "test_oracle_pins_rmsnorm.py::test_rmsnorm_eps_sits_inside_the_root"),
    ("rmsnorm_mean_511", "float mean = rmsnorm_sum_of_squares(x) / 512.0f;",
     "float mean = rmsnorm_sum_of_squares(x) / 511.0f;",
     "test_oracle_pins_rmsnorm.py::test_rmsnorm_matches_float64_within_one_ulp"),
    ("rmsnorm_weight_dropped", "float yw = bf16_to_f32(y) * bf16_to_f32(w[j]);",
     "float yw = bf16_to_f32(y);",
     "test_oracle_pins_rmsnorm.py::test_rmsnorm_weight_power_of_two_scales_exactly"),
    ("rmsnorm_y_unrounded", "float yw = bf16_to_f32(y) * bf16_to_f32(w[j]);",
     "float yw = xr * bf16_to_f32(w[j]); (void)y;",
     "test_oracle_pins_rmsnorm.py::test_rmsnorm_matches_float64_within_one_ulp"),
    ("rmsnorm_runs_of_16",
     "static int rmsnorm_block_element(int k, int i) { return i < 8 ? 8 * k + i : 256 + 8 * k + (i - 8); }",
     "static int rmsnorm_block_element(int k, int i) { return 16 * k + i; }",
     "test_oracle_pins_rmsnorm.py::test_rmsnorm_summation_order_golden"),
    ("rmsnorm_left_to_right",
     "        for (int k = 0; k < n / 2; ++k) sums[k] = sums[2 * k] + sums[2 * k + 1];\n    return sums[0];",
     "        ;\n    { float a = 0.0f; for (int j = 0; j < 512; ++j) { float v = bf16_to_f32(x[j]); "
     "a = a + v * v; } return a; }",
     "test_oracle_pins_rmsnorm.py::test_rmsnorm_summation_order_golden"),
    ("gather_scale_byte", "uint8_t scale_byte = row[latent_dim / 2 + j / group];",
     "uint8_t scale_byte = row[latent_dim / 2 + j / group] + 1;",
     "test_oracle_pins_store.py::test_gather_equals_independent_decode"),
    ("slot_upper_bound", "if (slot < 0 || slot >= num_slots) continue;",
     "if (slot < 0) continue;",
     "test_oracle_pins_store.py::test_store_skips_pads_and_out_of_range_and_keeps_poison"),
    ("block_stride_ignored", "return (block * block_stride_rows + row_in_block) * row_bytes;",
     "return (block * block_size + row_in_block) * row_bytes;",
     "test_oracle_pins_store.py::test_store_paged_addressing_with_block_stride"),
    ("amax_keeps_nan", "if (a > amax) amax = a;", "if (a > amax || a != a) amax = a;",
     "test_oracle_pins_store.py::test_store_worked_row"),
    # remaining insert layouts and save_ring_rows
    ("plain_nope_through_formula",
     "uint16_t h = j < 448 ? src[j] : f32_to_bf16_rne(rotated[j]);",
     "uint16_t h = f32_to_bf16_rne(rotated[j]);",
     "test_oracle_pins_inserts.py::test_plain_bf16_copies_nope_bits_and_rounds_rotary_values"),
    ("plain_fp8_reciprocal", "float y = x / fp8_scale;", "float y = x * (1.0f / fp8_scale);",
     "test_oracle_pins_inserts.py::test_plain_fp8_divides_by_the_scale"),
    ("v4_pad_scale", "scales[7] = 0;", "scales[7] = 127;",
     "test_oracle_pins_inserts.py::test_v4_record_layout_and_values"),
    ("v4_tile_32", "const int kTile = 64;", "const int kTile = 32;",
     "test_oracle_pins_inserts.py::test_v4_tiles_are_64_wide"),
    ("v4_bf16_byte_order", "values[448 + 2 * j] = (uint8_t)(h & 0xFF);",
     "values[448 + 2 * j] = (uint8_t)(h >> 8);",
     "test_oracle_pins_inserts.py::test_v4_record_layout_and_values"),
    ("ring_upper_bound", "if (slot < 0 || slot >= num_blocks * state_block) continue;",
     "if (slot < 0) continue;",
     "test_oracle_pins_inserts.py::test_ring_rows_copied_bit_for_bit_pads_skipped_slack_untouched"),
    # sparse attention (oracle/attention.py)
    ("attn_scale_dropped", "s = float(sm_scale) * (_bf16_to_f64(q[n]) @ k.T)",
     "s = (_bf16_to_f64(q[n]) @ k.T)",
     "test_oracle_pins_attention.py::test_two_keys_give_the_logistic_weights", "attention.py"),
    ("attn_pads_as_zero_rows", "valid = idx[n][(idx[n] >= 0) & (idx[n] < num_slots)]",
     "valid = np.where((idx[n] >= 0) & (idx[n] < num_slots), idx[n], -1)",
     "test_oracle_pins_attention.py::test_pads_are_dropped_and_order_does_not_matter",
     "attention.py"),
    ("attn_max_over_keys_axis", "m = s.max(axis=1, keepdims=True)",
     "m = s.max(axis=0, keepdims=True)",
     "test_oracle_pins_attention.py::test_brute_force_loops_on_a_tiny_case", "attention.py"),
    ("attn_lse_without_max", "lse[n] = m[:, 0] + np.log(l[:, 0])", "lse[n] = np.log(l[:, 0])",
     "test_oracle_pins_attention.py::test_single_valid_key_returns_its_row", "attention.py"),
    ("attn_abs_values", "out[n] = (p @ k) / l", "out[n] = (p @ np.abs(k)) / l",
     "test_oracle_pins_attention.py::test_single_valid_key_returns_its_row", "attention.py"),
    # fused_save_compress_norm (oracle/compress.py)
    ("fscn_ring_row_of_p", "state[s // cap, (int(pos[i]) - 1) % cap, :2 * LATENT]",
     "state[s // cap, int(pos[i]) % cap, :2 * LATENT]",
     "test_oracle_pins_compress.py::test_cr2_equals_streaming_model_and_is_invariant_to_chunking",
     "compress.py"),
    ("fscn_softmax_sign", "e0, e1 = np.exp(s0 - m), np.exp(s1 - m)",
     "e0, e1 = np.exp(m - s0), np.exp(m - s1)",
     "test_oracle_pins_compress.py::test_cr2_score_gap_sets_the_weights", "compress.py"),
    ("fscn_saves_first_rows", "for i in range(max(qs, qe - cap), qe):",
     "for i in range(qs, min(qe, qs + cap)):",
     "test_oracle_pins_compress.py::"
     "test_ring_save_takes_only_the_last_capacity_rows_and_skips_with_prev_rows", "compress.py"),
    ("fscn_saves_with_prev_rows", "if R == 2 and prev_rows is None:", "if R == 2:",
     "test_oracle_pins_compress.py::"
     "test_ring_save_takes_only_the_last_capacity_rows_and_skips_with_prev_rows", "compress.py"),
    ("fscn_prev_row_off_by_one", "j = int(prev_row_indices[k])",
     "j = int(prev_row_indices[k]) - 1",
     "test_oracle_pins_compress.py::test_prev_rows_select_the_predecessor", "compress.py"),
    ("fscn_eps_outside_root",
     "r = 1.0 / np.sqrt(np.mean(pooled * pooled, axis=1) + eps)",
     "r = 1.0 / (np.sqrt(np.mean(pooled * pooled, axis=1)) + eps)",
     "test_oracle_pins_compress.py::test_cr1_constant_row_closed_form", "compress.py"),
    ("fscn_closes_even_positions", "written = (slot >= 0) & (pos >= 0) & ((pos + 1) % R == 0)",
     "written = (slot >= 0) & (pos >= 0) & (pos % R == 0)",
     "test_oracle_pins_compress.py::test_cr2_equals_streaming_model_and_is_invariant_to_chunking",
     "compress.py"),
    ("fscn_weight_dropped", "latent = pooled * r[:, None] * w[None, :]",
     "latent = pooled * r[:, None]",
     "test_oracle_pins_compress.py::test_cr1_weight_and_alternating_signs", "compress.py"),
    ("bf16_nan_keeps_sign", "if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0u;",
     "if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u);",
     "test_oracle_pins_inserts.py::test_rotated_nan_is_stored_as_the_canonical_bf16_nan"),
    ("bf16_ties_away", "if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;",
     "if (lower >= 0x8000u) upper += 1u;",
     "test_oracle_pins_rmsnorm.py::test_rmsnorm_matches_float64_within_one_ulp"),
    ("nvfp4_scale_cap_240", "const float kMaxScale = 448.0f;", "const float kMaxScale = 240.0f;",
     "test_oracle_pins_rope.py::test_nvfp4_scale_clamps_to_448"),
    ("mxfp8_value_clamp_dropped", "        if (y > 448.0f) y = 448.0f;\n        if (y < -448.0f) y = -448.0f;\n        values[j] = oracle_e4m3_encode(y);",
     "        values[j] = oracle_e4m3_encode(y);",
     "test_oracle_pins_rope.py::test_mxfp8_scale_cap_depends_on_sanitising"),
    ("fscn_chunk_start_not_cut", "qs_t = np.maximum(qsl[r_safe], 0)", "qs_t = qsl[r_safe]",
     "test_oracle_pins_compress.py::test_cr2_chunk_bounds_are_cut_to_the_batch", "compress.py"),
]


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pin_catches_planted_mistake(tmp_path, mutant):
    name, orig, mutated, pin = mutant[:4]
    target = mutant[4] if len(mutant) > 4 else "kvq_oracle.c"
    src = open(os.path.join(ROOT, "oracle", target)).read()
    assert src.count(orig) == 1, f"{name}: the text to mutate is not unique in the oracle"
    shutil.copytree(os.path.join(ROOT, "oracle"), tmp_path / "oracle",
                    ignore=shutil.ignore_patterns("*.so", "__pycache__", "*.tmp*"))
    (tmp_path / "oracle" / target).write_text(src.replace(orig, mutated))
    shutil.copytree(os.path.join(ROOT, "tests"), tmp_path / "tests",
                    ignore=shutil.ignore_patterns("__pycache__", "test_*.py"))
    shutil.copy(os.path.join(ROOT, "tests", pin.split("::")[0]), tmp_path / "tests")
    shutil.copy(os.path.join(ROOT, "workloads.py"), tmp_path)
    env = dict(os.environ, PYTHONPATH=str(tmp_path))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        f"tests/{pin}"], cwd=tmp_path, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 1, f"{name} was not caught by {pin}:\n{r.stdout[-2000:]}"
