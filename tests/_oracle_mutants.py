"""Planted mistakes for the CPU oracle: evidence that its pins pin it.

Each entry names one oracle function and a small edit of its source -- a
dropped term, a wrong sign, index or axis, a swapped operand, an off-by-one
bound, the wrong constant -- of the kind a restatement of the pages could
plausibly contain. tests/test_oracle_mutants_cpu.py runs the oracle's pin
files once per entry, with this module loaded as a pytest plugin
(`-p _oracle_mutants`) and the entry's name in BEAM_ORACLE_MUTANT, and
expects the pins to fail every time.

The edit is made to a copy of the oracle's source text in memory, executed
into the oracle module's namespace in this process only; nothing on disk
changes and nothing outside the test process sees it.
"""
import os
import re

ENV = "BEAM_ORACLE_MUTANT"

# name -> (function, text in that function, replacement)
MUTANTS = {
    # elementwise helpers
    "bf16_truncates": ("bf16_round", "u + np.uint64(0x7FFF) + lsb", "u"),
    "bf16_ties_away": ("bf16_round", "u + np.uint64(0x7FFF) + lsb", "u + np.uint64(0x8000)"),
    "sigmoid_sign": ("sigmoid", "np.exp(-z)", "np.exp(z)"),
    "silu_no_z": ("silu", "return z * sigmoid(z)", "return sigmoid(z)"),
    "rms_eps_outside": ("rms_norm", "np.sqrt(ms + eps)", "(np.sqrt(ms) + eps)"),
    "rms_wrong_axis": ("rms_norm", "axis=-1", "axis=0"),
    "rms_gain_dropped": ("rms_norm", "out = out * np.asarray(gain, dtype=F64)", "out = out"),
    # router
    "bias_subtracted": ("router_scores", "logits + np.asarray(bias", "logits - np.asarray(bias"),
    "bias_after_sigmoid": ("router_scores", "s64 = sigmoid(logits)",
                           "s64 = sigmoid(x @ w.T) + (0 if bias is None else "
                           "np.asarray(bias, dtype=F64)[None, :])"),
    "group_top1": ("group_scores", "srt[..., 0] + srt[..., 1]", "srt[..., 0] + srt[..., 0]"),
    "group_top3": ("group_scores", "srt[..., 0] + srt[..., 1]",
                   "srt[..., 0] + srt[..., 1] + srt[..., 2]"),
    "ties_to_higher_index": ("_rank_desc", "np.lexsort((idx,", "np.lexsort((-idx,"),
    "no_group_limit": ("group_limited_topk", "for g in sorted(kept[t])", "for g in range(n_group)"),
    "one_group_too_few": ("group_limited_topk", "for g in sorted(kept[t])",
                          "for g in sorted(kept[t][:-1])"),
    "ascending_output": ("group_limited_topk", "idx[t] = corder[:top_k]",
                         "idx[t] = corder[:top_k][::-1]"),
    "scale_dropped": ("combine_weights", "return scale * sel /", "return sel /"),
    "normalised_over_all": ("combine_weights", "sel.sum(axis=1, keepdims=True)",
                            "s.sum(axis=1, keepdims=True)"),
    "topk_group_ignored": ("route", "group_limited_topk(s32, n_group, topk_group, top_k)",
                           "group_limited_topk(s32, n_group, n_group, top_k)"),
    "near_ties_needs_both": ("near_ties", ") | (", ") & ("),
    "groups_ranked_ascending": ("group_limited_topk", "gorder = _rank_desc(gs[t])",
                                "gorder = _rank_desc(-gs[t])"),
    # permutation
    "offsets_exclusive_shift": ("permutation", "np.cumsum(counts)]", "np.cumsum(counts) - counts]"),
    "pairs_by_token": ("permutation", "np.argsort(flat, kind=\"stable\")",
                       "np.arange(flat.size)"),
    "unstable_pair_order": ("permutation", "kind=\"stable\"", "kind=\"quicksort\""),
    # experts and combine
    "gate_up_swapped": ("swiglu_expert", "a = silu(g) * u", "a = silu(u) * g"),
    "silu_dropped": ("swiglu_expert", "a = silu(g) * u", "a = g * u"),
    "combine_unweighted": ("moe_combine", "out[tok] += weights[tok, slot][:, None] * y",
                           "out[tok] += y"),
    # residual stream
    "add_weight_not_sqrt": ("residual_coeffs", "1.0 / math.sqrt(k)", "1.0 / k"),
    "keep_weight_not_sqrt": ("residual_coeffs", "math.sqrt((k - 1) / k),", "(k - 1) / k,"),
    "post_norm_dropped": ("residual_step", "n = rms_norm(sub_out, gain, eps) if apply_norm",
                          "n = np.asarray(sub_out, F64) if apply_norm"),
    "coeffs_swapped": ("residual_step", "return a * np.asarray(h_prev, dtype=F64) + b * n",
                       "return b * np.asarray(h_prev, dtype=F64) + a * n"),
    "moe_residual_from_normed": ("moe_forward", "residual_step(x_in, out,", "residual_step(x, out,"),
    "moe_prenorm_gain_dropped": ("moe_forward", "rms_norm(x_in, pre_gain, eps)",
                                 "rms_norm(x_in, None, eps)"),
    "dense_residual_from_normed": ("dense_mlp_forward", "residual_step(x_in, y,",
                                   "residual_step(x, y,"),
    "post_gain_dropped": ("residual_step", "rms_norm(sub_out, gain, eps)",
                          "rms_norm(sub_out, None, eps)"),
    "moe_post_gain_dropped": ("moe_forward", "residual_k, post_gain, eps", "residual_k, None, eps"),
    "dense_prenorm_gain_dropped": ("dense_mlp_forward", "rms_norm(x_in, pre_gain, eps)",
                                   "rms_norm(x_in, None, eps)"),
    "rms_uses_mean_abs": ("rms_norm", "np.mean(v * v,", "np.mean(np.abs(v),"),
    # E4M3
    "e4m3_no_subnormal_floor": ("e4m3_round", "np.maximum(ex - 1, -6)", "(ex - 1)"),
    "e4m3_two_mantissa_bits": ("e4m3_round", "np.ldexp(1.0, e - 3)", "np.ldexp(1.0, e - 2)"),
    "e4m3_no_saturation": ("e4m3_round", "r = np.minimum(r, E4M3_MAX)", "r = r"),
    "e4m3_decode_bias_8": ("_e4m3_value", "np.ldexp(1.0, e - 7)", "np.ldexp(1.0, e - 8)"),
    "e4m3_decode_subnormal_step": ("_e4m3_value", "m * 2.0 ** -9", "m * 2.0 ** -10"),
    "e4m3_encode_bias_8": ("e4m3_encode", "e_unb + 7", "e_unb + 8"),
    "e4m3_scale_inverted": ("quantize_rows_e4m3", "np.where(nz, safe / F32(E4M3_MAX)",
                            "np.where(nz, F32(E4M3_MAX) / safe"),
    "e4m3_max_240": ("quantize_rows_e4m3", "inv = np.where(nz, F32(E4M3_MAX) / safe",
                     "inv = np.where(nz, F32(240.0) / safe"),
    "fp8_act_not_bf16": ("swiglu_expert_fp8", "a = bf16_round(swiglu_act_fp8(x_rows, gate_q, up_q))",
                         "a = swiglu_act_fp8(x_rows, gate_q, up_q)"),
    "fp8_x_not_quantised": ("swiglu_act_fp8", "xd = dequantize_rows_e4m3(qx, sx)",
                            "xd = np.asarray(x_rows, dtype=F64)"),
    "e4m3_decode_sign_flipped": ("e4m3_decode", "np.asarray(codes, dtype=np.uint8)]",
                                 "np.asarray(codes, dtype=np.uint8) ^ 0x80]"),
    "e4m3_dequant_divides": ("dequantize_rows_e4m3", "* np.asarray(scale", "/ np.asarray(scale"),
    "fp8_combine_unweighted": ("moe_combine_fp8", "out[tok] += weights[tok, slot][:, None] * y",
                               "out[tok] += y"),
    "fp8_residual_from_normed": ("moe_forward_fp8", "residual_step(x_in, out,",
                                 "residual_step(x, out,"),
    "e4m3_ties_away": ("e4m3_round", "np.round(a / q) * q", "np.floor(a / q + 0.5) * q"),
    "fp8_prenorm_gain_dropped": ("moe_forward_fp8", "rms_norm(x_in, pre_gain, eps)",
                                 "rms_norm(x_in, None, eps)"),
    "fp8_post_gain_dropped": ("moe_forward_fp8", "residual_k, post_gain, eps",
                              "residual_k, None, eps"),
    # E2M1 / NVFP4
    "e2m1_half_steps_below_one": ("e2m1_round", "np.clip(ex - 1, 0, 2)", "np.clip(ex - 1, -1, 2)"),
    "e2m1_no_saturation": ("e2m1_round", "np.minimum(np.where(a == 0, 0.0, r), E2M1_MAX)",
                           "np.where(a == 0, 0.0, r)"),
    "e2m1_decode_exponent": ("e2m1_decode", "np.ldexp(1.0, e - 1)", "np.ldexp(1.0, e)"),
    "nibbles_swapped": ("pack_e2m1", "(c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)",
                        "(c[..., 1::2] & 0xF) | ((c[..., 0::2] & 0xF) << 4)"),
    "nvfp4_group_scale_448": ("quantize_nvfp4", "amax / F32(2688.0)", "amax / F32(448.0)"),
    "nvfp4_block_scale_no_6": ("quantize_nvfp4", "six_g = (F32(6.0) * g_row)", "six_g = (g_row)"),
    "nvfp4_group_scale_dropped": ("dequantize_nvfp4", "* g[:, None, None]", "* 1.0"),
    "nvfp4_gate_up_swapped": ("swiglu_act_nvfp4", "return silu(g) * u", "return silu(u) * g"),
    "e2m1_encode_sign_bit_2": ("e2m1_encode", "<< np.uint8(3)", "<< np.uint8(2)"),
    "unpack_nibbles_swapped": ("unpack_e2m1", "out[..., 0::2] = p & 0xF\n    out[..., 1::2] = p >> 4",
                               "out[..., 0::2] = p >> 4\n    out[..., 1::2] = p & 0xF"),
    "nvfp4_act_not_bf16": ("swiglu_expert_nvfp4",
                           "a = bf16_round(swiglu_act_nvfp4(x_rows, gate_q, up_q))",
                           "a = swiglu_act_nvfp4(x_rows, gate_q, up_q)"),
    "nvfp4_combine_unweighted": ("moe_combine_nvfp4",
                                 "out[tok] += weights[tok, slot][:, None] * swiglu_expert_nvfp4(",
                                 "out[tok] += swiglu_expert_nvfp4("),
    "e2m1_ties_away": ("e2m1_round", "np.round(a / q) * q", "np.floor(a / q + 0.5) * q"),
    # attention
    "rope_sin_sign": ("rope_rotate", "x2 * cos + x1 * sin", "x2 * cos - x1 * sin"),
    "rope_frequency_halved": ("rope_rotate", "* 2.0 / d)", "/ d)"),
    "rope_interleaved_pairs": ("rope_rotate", "x1, x2 = v[..., :half], v[..., half:]",
                               "x1, x2 = v[..., 0::2], v[..., 1::2]"),
    "query_scale_power": ("global_query_scale", "** 0.1", "** 0.5"),
    "query_scale_pos_not_plus_one": ("global_query_scale", "np.asarray(pos, dtype=F64) + 1.0",
                                     "np.asarray(pos, dtype=F64)"),
    "window_off_by_one": ("attention_core", "(i - j) < window", "(i - j) <= window"),
    "softmax_scale_1_over_d": ("attention_core", "/ math.sqrt(d)", "/ d"),
    "gqa_heads_interleaved": ("attention_core", "h // group", "h % k.shape[0]"),
    "gate_not_sigmoid": ("attention_forward", "gate = sigmoid(qg[:, dq:])", "gate = qg[:, dq:]"),
    "q_norm_uses_k_gain": ("attention_forward", "q = rms_norm(q, q_gain, eps)",
                           "q = rms_norm(q, k_gain, eps)"),
    "norm_after_position": ("attention_forward",
                            "q = rms_norm(q, q_gain, eps)\n    k = rms_norm(k, k_gain, eps)\n"
                            "    if window > 0:\n"
                            "        q = rope_rotate(q, rows, rope_theta)\n"
                            "        k = rope_rotate(k, np.arange(T), rope_theta)\n"
                            "    else:\n"
                            "        q = q * global_query_scale(rows)[None, :, None]\n",
                            "if window > 0:\n"
                            "        q = rope_rotate(q, rows, rope_theta)\n"
                            "        k = rope_rotate(k, np.arange(T), rope_theta)\n"
                            "    else:\n"
                            "        q = q * global_query_scale(rows)[None, :, None]\n"
                            "    q = rms_norm(q, q_gain, eps)\n    k = rms_norm(k, k_gain, eps)\n"),
    "causal_excludes_self": ("attention_core", "allowed = j <= i", "allowed = j < i"),
    "k_v_swapped": ("attention_forward", "k = kv[:, :dkv]", "k = kv[:, dkv:]"),
    "attn_residual_from_normed": ("attention_forward", "residual_step(h_in[rows], out,",
                                  "residual_step(x[rows], out,"),
    "attn_prenorm_gain_dropped": ("attention_forward", "rms_norm(h_in, pre_gain, eps)",
                                  "rms_norm(h_in, None, eps)"),
    "attn_post_gain_dropped": ("attention_forward", "residual_k, post_gain, eps",
                               "residual_k, None, eps"),
    "bf16_mask_drops_bit": ('bf16_round', 'np.uint64(0xFFFF0000)', 'np.uint64(0xFFFE0000)'),
    "group_margin_wrong_rank": ('group_limited_topk', 'gorder[topk_group - 1]', 'gorder[topk_group - 2]'),
    "topk_margin_wrong_rank": ('group_limited_topk', 'corder[top_k - 1]', 'corder[top_k - 2]'),
    "e4m3_sign_dropped": ('e4m3_round', 'return np.copysign(r, v)', 'return r'),
    "e4m3_encode_subnormal_step": ('e4m3_encode', 'm_sub = a / 2.0 ** -9', 'm_sub = a / 2.0 ** -10'),
    "e4m3_top_binade_is_nan": ('_e4m3_value', '(e == 15) & (m == 7)', '(e == 15)'),
    "nvfp4_group_scales_tiled": ('quantize_nvfp4', 'np.repeat(g, rows_per_group)', 'np.tile(g, rows_per_group)'),
    "nvfp4_multiplies_by_scale": ('quantize_nvfp4', 'F32(1.0) / np.where(sb_val > 0, denom, F32(1.0))', 'np.where(sb_val > 0, denom, F32(1.0))'),
    "nvfp4_dequant_group_tiled": ('dequantize_nvfp4', 'np.repeat(np.asarray(group_scales, dtype=F64), rows_per_group)', 'np.tile(np.asarray(group_scales, dtype=F64), rows_per_group)'),
    "nvfp4_x_not_quantised": ('swiglu_act_nvfp4', 'xd = dequantize_nvfp4(*quantize_nvfp4(x_rows, 1), 1)', 'xd = np.asarray(x_rows, dtype=F64)'),
    "nvfp4_act_not_quantised": ('swiglu_expert_nvfp4', 'ad = dequantize_nvfp4(*quantize_nvfp4(a, 1), 1)', 'ad = np.asarray(a, dtype=F64)'),
    "fp8_act_not_quantised": ('swiglu_expert_fp8', 'return dequantize_rows_e4m3(qa, sa) @', 'return np.asarray(a, dtype=F64) @'),
    "softmax_normalised_over_queries": ('attention_core', 'p / p.sum(axis=1, keepdims=True)', 'p / p.sum(axis=0, keepdims=True)'),
    "query_scale_relative_rows": ('attention_forward', 'global_query_scale(rows)', 'global_query_scale(np.arange(len(rows)))'),
    "gate_after_rounding": ('attention_forward', 'bf16_round(o.transpose(1, 0, 2).reshape(len(rows), dq) * gate)', 'bf16_round(o.transpose(1, 0, 2).reshape(len(rows), dq)) * gate'),
    "forward_ignores_window": ('attention_forward', 'attention_core(q, k, v, window, q_pos=rows)', 'attention_core(q, k, v, 0, q_pos=rows)'),
    "v_not_rounded": ("attention_forward", "q, k, v = (bf16_round(a).astype(F64) for a in (q, k, v))",
                      "q, k = (bf16_round(a).astype(F64) for a in (q, k))"),
    "residual_allows_k1": ('residual_coeffs', 'if k < 2:', 'if k < 1:'),
}


def function_span(src, name):
    """(start, end) of the top-level `def name(` block in src: from its def
    line to the next line that starts at column 0 with anything but a
    closing bracket."""
    m = re.search(r"^def " + re.escape(name) + r"\(", src, flags=re.M)
    if m is None:
        raise KeyError(f"no top-level function {name}")
    nxt = re.compile(r"^[^\s)]", flags=re.M).search(src, m.end())
    return m.start(), (nxt.start() if nxt else len(src))


def mutated_source(src, name):
    """The oracle source with the edit of MUTANTS[name] made inside its function."""
    fn, old, new = MUTANTS[name]
    a, b = function_span(src, fn)
    body = src[a:b]
    if old not in body:
        raise ValueError(f"mutant {name}: text not found in {fn}")
    return src[:a] + body.replace(old, new) + src[b:]


def apply(name):
    """Execute the mutated oracle source into the oracle module's namespace
    and re-export its public names from the `oracle` package."""
    import oracle
    import oracle.beam_oracle as M
    with open(M.__file__, encoding="utf-8") as f:
        src = f.read()
    exec(compile(mutated_source(src, name), M.__file__, "exec"), M.__dict__)
    for k, v in M.__dict__.items():
        if not k.startswith("_") and hasattr(oracle, k):
            setattr(oracle, k, v)


def pytest_configure(config):
    name = os.environ.get(ENV)
    if name:
        apply(name)
