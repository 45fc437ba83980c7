"""The oracle's pins are strong enough to catch plausible mistakes.

Each case below plants one mistake in a private copy of the oracle's source
(a dropped term, a flipped sign, an off-by-one exponent or bias, a wrong
index or operand, a wrong rounding rule) and runs the pins of
test_oracle_encodings.py and test_oracle_path.py against that copy: at least
one pin has to fail.  The unmodified copy has to pass all of them, which
checks the harness itself.  Nothing here touches the oracle that the other
tests import.
"""

import pytest

from pins_harness import failing_pins, oracle_copy

ROPE_X0 = "x0 = x_f32[t, :, D - R:D - half].astype(np.float32)"
ROPE_X1 = "x1 = x_f32[t, :, D - half:D].astype(np.float32)"
ROPE_Y0 = "y[t, :, D - R:D - half] = (x0 * c) + (x1 * s)"
ROPE_Y1 = "y[t, :, D - half:D] = (x1 * c) - (x0 * s)"

# (name, [(text in the oracle, replacement), ...]); every text occurs once.
MISTAKES = [
    # E4M3 decode
    ("e4m3_subnormal_quantum_2^-10", [("mag = M * 2.0 ** -9", "mag = M * 2.0 ** -10")]),
    ("e4m3_exponent_bias_8", [("2.0 ** (E - 7)\n    return -mag", "2.0 ** (E - 8)\n    return -mag")]),
    ("e4m3_mantissa_over_16", [("(1.0 + M / 8.0)", "(1.0 + M / 16.0)")]),
    ("e4m3_no_nan_code", [("if E == 0xF and M == 0x7:", "if False:")]),
    # E4M3 encode
    ("encode_ties_away_from_zero", [("& (_POS_CODES[lo] % 2 == 0))", "& False)")]),
    ("encode_ties_to_odd", [("_POS_CODES[lo] % 2 == 0", "_POS_CODES[lo] % 2 == 1")]),
    ("encode_truncates", [("pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (_POS_CODES[lo] % 2 == 0))",
                           "pick_lo = d_hi > 0")]),
    ("encode_overflow_to_nan", [("np.where(a >= E4M3_MAX, 0x7E, code)", "np.where(a > E4M3_MAX, 0x7F, code)")]),
    ("encode_nan_not_kept", [("    code = np.where(np.isnan(v), 0x7F, code)\n", "")]),
    ("encode_drops_sign_of_zero", [("code | np.where(neg, 0x80, 0)", "code | np.where(neg & (code != 0), 0x80, 0)")]),
    # E8M0 scale rule
    ("scale_threshold_inclusive", [("(m > 0.875)", "(m >= 0.875)")]),
    ("scale_exponent_off_by_one", [("- 9 + (m > 0.875)", "- 8 + (m > 0.875)")]),
    ("scale_max_256_not_448", [("(m > 0.875)", "(m > 0.5)")]),
    ("scale_zero_group_not_min", [("e = np.where(amax == 0.0, -127, e)", "pass")]),
    ("scale_not_clamped", [("return np.clip(e, -127, 127)", "return e")]),
    # inverse RoPE
    ("rope_forward_not_inverse", [(ROPE_Y0, ROPE_Y0.replace("+ (x1", "- (x1")),
                                  (ROPE_Y1, ROPE_Y1.replace("- (x0", "+ (x0"))]),
    ("rope_on_first_R_elements", [(ROPE_X0, "x0 = x_f32[t, :, 0:half].astype(np.float32)"),
                                  (ROPE_X1, "x1 = x_f32[t, :, half:R].astype(np.float32)"),
                                  (ROPE_Y0, ROPE_Y0.replace("D - R:D - half", "0:half")),
                                  (ROPE_Y1, ROPE_Y1.replace("D - half:D", "half:R"))]),
    ("rope_interleaved_pairs", [(ROPE_X0, "x0 = x_f32[t, :, D - R:D:2].astype(np.float32)"),
                                (ROPE_X1, "x1 = x_f32[t, :, D - R + 1:D:2].astype(np.float32)"),
                                (ROPE_Y0, ROPE_Y0.replace("D - R:D - half", "D - R:D:2")),
                                (ROPE_Y1, ROPE_Y1.replace("D - half:D", "D - R + 1:D:2"))]),
    ("rope_cos_sin_swapped", [(ROPE_Y0, "y[t, :, D - R:D - half] = (x0 * s) + (x1 * c)"),
                              (ROPE_Y1, "y[t, :, D - half:D] = (x1 * s) - (x0 * c)")]),
    ("rope_table_row_by_token", [("p = int(pos[t])", "p = t")]),
    ("rope_half_fixed_at_32", [("half = R // 2", "half = 32")]),
    ("rope_output_rounded_to_bf16", [("        y[t, :, D - half:D] = (x1 * c) - (x0 * s)\n    return y",
                                      "        y[t, :, D - half:D] = (x1 * c) - (x0 * s)\n"
                                      "    return bf16_bits_to_f32(bf16_rne_bits(y.astype(np.float64)))")]),
    ("rope_skipped", [("y = inverse_rope_rows(x, pos, cos_bits, sin_bits, R)", "y = x")]),
    # group quantisation
    ("quant_scale_bias_128", [("scales[..., kg] = (e + 127)", "scales[..., kg] = (e + 128)")]),
    ("quant_multiplies_by_scale", [("np.ldexp(blk, -e[..., None])", "np.ldexp(blk, e[..., None])")]),
    ("quant_signed_amax", [("np.max(np.abs(blk), axis=-1)", "np.max(blk, axis=-1)")]),
    ("quant_group_64", [("GROUP = 128", "GROUP = 64")]),
    ("quant_amax_over_whole_row", [("amax = np.max(np.abs(blk), axis=-1)",
                                    "amax = np.max(np.abs(y.astype(np.float64)), axis=-1)")]),
    # MX values, dequantisation
    ("scale_index_k_mod_groups", [("np.repeat(np.asarray(scales), GROUP, axis=-1)",
                                   "np.tile(np.asarray(scales), GROUP)")]),
    ("e8m0_bias_128", [("sc - 127)", "sc - 128)")]),
    ("e8m0_ff_not_nan", [("return np.where(sc == 255, np.nan, val)", "return val")]),
    ("bf16_truncates", [("n = np.rint(np.ldexp(a, -q))", "n = np.floor(np.ldexp(a, -q))")]),
    ("bf16_no_subnormal_quantum", [("q = np.maximum(E.astype(np.int64) - 8, -133)", "q = E.astype(np.int64) - 8")]),
    ("bf16_nine_bits", [("q = np.maximum(E.astype(np.int64) - 8, -133)", "q = np.maximum(E.astype(np.int64) - 9, -133)")]),
    # GEMM
    ("gemm_first_group_weight_for_all", [("A[:, g, :] @ W[g].T", "A[:, g, :] @ W[0].T")]),
    ("gemm_weight_read_as_k_by_n", [("A[:, g, :] @ W[g].T", "A[:, g, :] @ W[g].reshape(K, N)")]),
    ("gemm_abs_sum_of_result", [("np.abs(A[:, g, :]) @ np.abs(W[g]).T", "np.abs(A[:, g, :] @ W[g].T)")]),
    ("gemm_abs_sum_drops_weight_abs", [("np.abs(A[:, g, :]) @ np.abs(W[g]).T", "np.abs(A[:, g, :]) @ W[g].T")]),
    ("linear_skips_activation_quant", [("    y, S = bmm_a8w8_ref(a_codes[:, None, :]",
                                        "    a_codes, a_scales = group_quant_rows(x.astype(np.float32) * 1.0)\n"
                                        "    a_scales = a_scales + 1\n"
                                        "    y, S = bmm_a8w8_ref(a_codes[:, None, :]")]),
    ("linear_uses_unquantised_x", [("    y, S = bmm_a8w8_ref(a_codes[:, None, :], a_scales[:, None, :],\n"
                                     "                        w_codes[None], w_scales[None])\n"
                                     "    return y[:, 0, :], S[:, 0, :], a_codes, a_scales",
                                     "    Wv = mx_values(w_codes, w_scales)\n"
                                     "    y = x.astype(np.float64) @ Wv.T\n"
                                     "    S = np.abs(x.astype(np.float64)) @ np.abs(Wv).T\n"
                                     "    return y, S, a_codes, a_scales")]),
    ("linear_partial_group_amax_over_128", [("    a_codes, a_scales = group_quant_rows(x)\n",
                                              "    a_codes, a_scales = group_quant_rows(x)\n"
                                              "    a_scales[:, -1] = np.maximum(a_scales[:, -1], a_scales[:, 0])\n")]),
    # forward RoPE and KV-cache insert
    ("fwd_rope_is_inverse", [("y[t, :, D - R:D - h] = (a * cs) - (b * sn)", "y[t, :, D - R:D - h] = (a * cs) + (b * sn)"),
                             ("y[t, :, D - h:D] = (b * cs) + (a * sn)", "y[t, :, D - h:D] = (b * cs) - (a * sn)")]),
    ("fwd_rope_cos_sin_swapped", [("y[t, :, D - R:D - h] = (a * cs) - (b * sn)", "y[t, :, D - R:D - h] = (a * sn) - (b * cs)")]),
    ("fwd_rope_table_row_by_token", [("row = int(pos[t])", "row = t")]),
    ("fwd_rope_pairs_adjacent", [("a = x_f32[t, :, D - R:D - h]", "a = x_f32[t, :, D - R:D:2]"),
                                 ("b = x_f32[t, :, D - h:D]", "b = x_f32[t, :, D - R + 1:D:2]"),
                                 ("y[t, :, D - R:D - h] = (a * cs) - (b * sn)", "y[t, :, D - R:D:2] = (a * cs) - (b * sn)"),
                                 ("y[t, :, D - h:D] = (b * cs) + (a * sn)", "y[t, :, D - R + 1:D:2] = (b * cs) + (a * sn)")]),
    ("kv_scale_multiplied", [("v = k / np.float32(scale)", "v = k * np.float32(scale)")]),
    ("kv_scale_in_fp64", [("v = k / np.float32(scale)", "v = k.astype(np.float64) / scale")]),
    ("kv_negative_slot_written", [("if int(slots[t]) >= 0:", "if True:")]),
    ("kv_not_rotated", [("k = forward_rope_rows(kv, pos, cos_bits, sin_bits, R)[:, 0, :]", "k = kv[:, 0, :]")]),
    ("q_not_rotated", [("q_out = bf16_rne_bits(forward_rope_rows(q, pos, cos_bits, sin_bits, R).astype(np.float64))",
                        "q_out = bf16_rne_bits(q.astype(np.float64))")]),
    ("q_rounded_before_rotation", [("    q = bf16_bits_to_f32(q_bits)\n",
                                    "    q = bf16_bits_to_f32(q_bits)\n    q = (q * np.float32(1.0000001)).astype(np.float32)\n")]),
    # tolerance, scale conversion
    ("ulp_off_by_one", [("ex = np.maximum(E.astype(np.int64) - 1, -126) - 7",
                         "ex = np.maximum(E.astype(np.int64) - 1, -126) - 8")]),
    ("tolerance_relative_1e-4", [("1e-5 * np.asarray(S", "1e-4 * np.asarray(S")]),
    ("f32_scale_accepts_non_powers", [("& (m == 0.5) ", "")]),
    ("f32_scale_accepts_negative", [("np.isfinite(s) & (s > 0) &", "np.isfinite(s) & (s != 0) &"),
                                    ("m, E = np.frexp(s)\n", "m, E = np.frexp(np.abs(s))\n")]),
    ("f32_scale_bias_128", [("np.where(ok, k + 127, 255)", "np.where(ok, k + 128, 255)")]),
    ("f32_scale_range_128", [("(k >= -127) & (k <= 127)", "(k >= -128) & (k <= 127)")]),
]


def test_unmodified_copy_passes_every_pin():
    assert failing_pins(oracle_copy([]), stop_at_first=False) == []


@pytest.mark.parametrize("edits", [m[1] for m in MISTAKES], ids=[m[0] for m in MISTAKES])
def test_planted_mistake_fails_a_pin(edits):
    assert failing_pins(oracle_copy(edits), stop_at_first=True), "no pin caught this mistake"
