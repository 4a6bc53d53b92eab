"""The oracle's pins are strong enough to catch plausible slips: each case below plants one
mistake in a copy of the oracle's source (on the CPU, in memory; the committed oracle is not
touched) and checks that at least one of the named pins fails on the mutant. A slip that no
pin catches would be a gap in the pins."""
import os
import types

import pytest

import oracle
import test_oracle_codecs as codec_pins
import test_oracle_pins as pins

SRC_PATH = os.path.join(os.path.dirname(oracle.__file__), "beam_oracle.py")
SRC = open(SRC_PATH).read()

# (slip, text in the oracle, planted text, pins that must catch it)
MUTATIONS = [
    ("RMSNorm drops its gain",
     "return x / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)",
     "return x / np.sqrt(ms + eps)",
     ["test_rmsnorm_unit_rms_and_scale_invariance"]),
    ("RMSNorm sums instead of averaging",
     "ms = np.mean(x * x, axis=-1, keepdims=True)",
     "ms = np.sum(x * x, axis=-1, keepdims=True)",
     ["test_rmsnorm_unit_rms_and_scale_invariance"]),
    ("residual coefficients swapped",
     "h = bf16_round(np.sqrt((n - 1.0) / n) * h + y / np.sqrt(n))",
     "h = bf16_round(np.sqrt(1.0 / n) * h + y * np.sqrt((n - 1.0) / n))",
     ["test_residual_first_term_and_coefficients", ("test_depth_scaled_residual_keeps_unit_variance", 3)]),
    ("residual adds without the depth scaling",
     "h = bf16_round(np.sqrt((n - 1.0) / n) * h + y / np.sqrt(n))",
     "h = bf16_round(h + y / np.sqrt(n))",
     [("test_depth_scaled_residual_keeps_unit_variance", 10), "test_residual_first_term_and_coefficients"]),
    ("sublayer output not post-normed",
     "y = bf16_round(rmsnorm(x, w_post, eps))",
     "y = bf16_round(x)",
     ["test_residual_first_term_and_coefficients"]),
    ("RoPE rotation sign flipped",
     "x2 * c + x1 * s], axis=-1)",
     "x2 * c - x1 * s], axis=-1)",
     ["test_rope_closed_forms", "test_rope_invariants"]),
    ("RoPE pairs adjacent elements instead of halves",
     "x1, x2 = x[..., :half], x[..., half:]",
     "x1, x2 = x[..., 0::2], x[..., 1::2]",
     ["test_rope_closed_forms", "test_rope_invariants"]),
    ("RoPE frequency exponent halved",
     "return np.power(float(theta), -2.0 * i / D)",
     "return np.power(float(theta), -1.0 * i / D)",
     ["test_rope_closed_forms"]),
    ("RoPE angle from p instead of p - 1",
     "m = (pos - 1)[:, None]",
     "m = pos[:, None]",
     ["test_qkv_gate_rope_relative_position", "test_rope_closed_forms"]),
    ("SSMax exponent sign",
     "return np.power(1.0 + np.asarray(p, dtype=np.float64) / base, expo)",
     "return np.power(1.0 + np.asarray(p, dtype=np.float64) / base, -expo)",
     ["test_ssmax_values"]),
    ("SSMax also scales k",
     "qn = qn * ssmax_scale(pos, cfg.ssmax_base, cfg.ssmax_exp)[:, None, None]",
     "qn = qn * ssmax_scale(pos, cfg.ssmax_base, cfg.ssmax_exp)[:, None, None]\n"
     "        kn = kn * ssmax_scale(pos, cfg.ssmax_base, cfg.ssmax_exp)[:, None, None]",
     ["test_qkv_gate_packed_row_order", "test_qkv_gate_nope_scales_q_only"]),
    ("cache slot p instead of p - 1",
     "return (np.asarray(p) - 1) % self.capacity",
     "return np.asarray(p) % self.capacity",
     ["test_kv_cache_ring_and_fp8_roundtrip"]),
    ("window one key too wide",
     "lo = 1 if cache.window == 0 else max(1, p - cache.window + 1)",
     "lo = 1 if cache.window == 0 else max(1, p - cache.window)",
     ["test_attention_special_cases", "test_attention_matches_torch_sdpa"]),
    ("softmax scale 1/D instead of 1/sqrt(D)",
     "logits = qh @ K[hk, a:b].T / np.sqrt(D)",
     "logits = qh @ K[hk, a:b].T / D",
     ["test_attention_matches_torch_sdpa"]),
    ("query attends to all but itself",
     "a, b = lo - lo_all, p - lo_all + 1",
     "a, b = lo - lo_all, max(p - lo_all, lo - lo_all + 1)",
     ["test_attention_matches_torch_sdpa", "test_attention_special_cases"]),
    ("softmax normalised over the query heads",
     "o[t, hk * grp:(hk + 1) * grp] = (e / e.sum(axis=1, keepdims=True)) @ V[hk, a:b]",
     "o[t, hk * grp:(hk + 1) * grp] = (e / e.sum(axis=0, keepdims=True)) @ V[hk, a:b]",
     ["test_attention_matches_torch_sdpa", "test_attention_special_cases"]),
    ("GQA heads interleaved instead of grouped",
     "qh = q[t, hk * grp:(hk + 1) * grp]",
     "qh = q[t, hk::Hkv]",
     ["test_attention_gqa_head_mapping_and_gate", "test_attention_matches_torch_sdpa"]),
    ("gate sigmoid sign flipped",
     "gate = 1.0 / (1.0 + np.exp(-(np.asarray(g, dtype=np.float64) + gb)))",
     "gate = 1.0 / (1.0 + np.exp(np.asarray(g, dtype=np.float64) + gb))",
     ["test_attention_gqa_head_mapping_and_gate"]),
    ("group score from the best expert only",
     "gscore = (top2[:, 0] + top2[:, 1]).astype(np.float32)",
     "gscore = (top2[:, 0] + top2[:, 0]).astype(np.float32)",
     ["test_route_matches_brute_force_tiny", "test_route_group_choice_full_width"]),
    ("routing weights from the biased scores",
     "ssel = s[t, sel].astype(np.float64)",
     "ssel = b[t, sel].astype(np.float64)",
     ["test_route_weights_use_unbiased_scores"]),
    ("routing weights without the 2.5 scale",
     "w[t] = ssel / ssel.sum() * cfg.route_scale",
     "w[t] = ssel / ssel.sum()",
     ["test_route_weights_use_unbiased_scores", "test_route_matches_brute_force_tiny"]),
    ("expert SwiGLU gate and up swapped",
     "return bf16_round(silu(gu[:F]) * gu[F:])",
     "return bf16_round(gu[:F] * silu(gu[F:]))",
     ["test_moe_equals_dense_with_stacked_experts"]),
    ("combine ignores the routing weights",
     "acc += float(w[t, j]) * y",
     "acc += y",
     ["test_moe_combine_is_weighted_sum"]),
    ("NoPE layers every 6th from layer 0",
     "return (layer + 1) % 6 == 0 or layer == n_layers - 1",
     "return layer % 6 == 0 or layer == n_layers - 1",
     ["test_layer_count_gives_104_boundaries"]),
    ("attention residual index 2l + 1",
     'h, u = boundary_norm(a, h, W["attn_post"], W["mlp_pre"], 2 * l + 2, cfg.eps)',
     'h, u = boundary_norm(a, h, W["attn_post"], W["mlp_pre"], 2 * l + 1, cfg.eps)',
     ["test_residual_index_counts_every_addition"]),
    ("gate and V rows of the packed projection swapped",
     "g = z[:, (Hq + 2 * Hkv) * D:]",
     "g = np.concatenate([z[:, (Hq + Hkv) * D: (Hq + 2 * Hkv) * D]] * (Hq // Hkv), axis=1)",
     ["test_qkv_gate_packed_row_order"]),
    ("K and V rows of the packed projection swapped",
     "k = z[:, Hq * D: (Hq + Hkv) * D].reshape(T, Hkv, D)\n"
     "    v = z[:, (Hq + Hkv) * D: (Hq + 2 * Hkv) * D].reshape(T, Hkv, D)",
     "v = z[:, Hq * D: (Hq + Hkv) * D].reshape(T, Hkv, D)\n"
     "    k = z[:, (Hq + Hkv) * D: (Hq + 2 * Hkv) * D].reshape(T, Hkv, D)",
     ["test_qkv_gate_packed_row_order", "test_qkv_gate_nope_scales_q_only"]),
    ("router scores by exp instead of sigmoid",
     "s = f32(1.0 / (1.0 + np.exp(-logits.astype(np.float64))))",
     "s = f32(np.exp(logits.astype(np.float64)))",
     ["test_route_weights_use_unbiased_scores", "test_route_matches_brute_force_tiny"]),
    ("dense SwiGLU gate and up swapped",
     "a = bf16_round(silu(gu[:, :Fd]) * gu[:, Fd:])",
     "a = bf16_round(gu[:, :Fd] * silu(gu[:, Fd:]))",
     ["test_moe_equals_dense_with_stacked_experts"]),
    ("FP8 cache store multiplies by the scale",
     "self.k[s, :, sl, :] = e4m3_encode(f32(k_vec) / np.float32(self.k_scale))",
     "self.k[s, :, sl, :] = e4m3_encode(f32(k_vec) * np.float32(self.k_scale))",
     ["test_kv_cache_ring_and_fp8_roundtrip"]),
    ("FP8 cache load divides by the scale",
     "return e4m3_decode(k) * self.k_scale, e4m3_decode(v) * self.v_scale",
     "return e4m3_decode(k) / self.k_scale, e4m3_decode(v) * self.v_scale",
     ["test_kv_cache_ring_and_fp8_roundtrip"]),
    ("expert ties go to the higher index",
     "corder = np.lexsort((cand, -b[t, cand].astype(np.float64)))",
     "corder = np.lexsort((-cand, -b[t, cand].astype(np.float64)))",
     ["test_route_ties_go_to_lower_index", "test_route_matches_brute_force_tiny", "test_route_group_choice_full_width",
      "test_route_weights_use_unbiased_scores"]),
    ("group ties go to the higher index",
     "gorder = np.lexsort((np.arange(G), -gscore.astype(np.float64)))",
     "gorder = np.lexsort((-np.arange(G), -gscore.astype(np.float64)))",
     ["test_route_ties_go_to_lower_index", "test_route_matches_brute_force_tiny", "test_route_group_choice_full_width",
      "test_route_weights_use_unbiased_scores"]),
    ("softcap without the division by c",
     "z = softcap * np.tanh(z / softcap)",
     "z = softcap * np.tanh(z)",
     ["test_lm_head_softcap_closed_forms"]),
    ("LM head projection transposed",
     "z = np.asarray(u, dtype=np.float64) @ np.asarray(w_lm, dtype=np.float64).T",
     "z = (np.asarray(w_lm, dtype=np.float64) @ np.asarray(u, dtype=np.float64).T).T[:, ::-1]",
     ["test_lm_head_projection_brute_force"]),
]


CODECS_PATH = os.path.join(os.path.dirname(oracle.__file__), "codecs.py")
CODECS_SRC = open(CODECS_PATH).read()

CODEC_MUTATIONS = [
    ("bf16 truncates",
     "r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)",
     "r = (u >> np.uint64(16)).astype(np.uint16)",
     ["test_bf16_encode_random_matches_torch"]),
    ("bf16 ties away from zero",
     "r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)",
     "r = ((u + np.uint64(0x8000)) >> np.uint64(16)).astype(np.uint16)",
     ["test_bf16_ties_go_to_even"]),
    ("e4m3 exponent bias 8",
     "vals[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)",
     "vals[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 8)",
     ["test_e4m3_decode_matches_torch_all_codes"]),
    ("e4m3 does not saturate",
     "q = np.minimum(q, E4M3_MAX)",
     "q = q",
     ["test_e4m3_saturates_and_keeps_nan"]),
    ("e4m3 subnormal binade misplaced",
     "e = np.maximum(e, -6.0)",
     "e = np.maximum(e, -7.0)",
     ["test_e4m3_encode_in_range_matches_torch"]),
    ("e2m1 subnormal step 1 instead of 0.5",
     "vals[code] = sign * (m * 0.5 if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1))",
     "vals[code] = sign * (m * 1.0 if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1))",
     ["test_e2m1_codes_are_the_published_magnitudes"]),
    ("NVFP4 nibble order swapped",
     "out[..., 0::2] = b & np.uint8(0xF)\n    out[..., 1::2] = b >> np.uint8(4)",
     "out[..., 1::2] = b & np.uint8(0xF)\n    out[..., 0::2] = b >> np.uint8(4)",
     ["test_nvfp4_nibble_order_block_and_matrix_scales"]),
    ("NVFP4 matrix scale dropped",
     "return v.reshape(rows, K) * float(np.float32(matrix_scale))",
     "return v.reshape(rows, K)",
     ["test_nvfp4_nibble_order_block_and_matrix_scales", "test_nvfp4_dequant_matches_element_loop"]),
    ("FP8 block scale ignored",
     "return v * s[rb[:, None], kb[None, :]]",
     "return v",
     ["test_fp8_block_scales_hand_built", "test_fp8_block_dequant_matches_element_loop"]),
    ("FP8 block scale indices transposed",
     "return v * s[rb[:, None], kb[None, :]]",
     "return v * s[kb[None, :], rb[:, None]]",
     ["test_fp8_block_scales_hand_built", "test_fp8_block_dequant_matches_element_loop"]),
]


def mutant(old, new):
    assert SRC.count(old) == 1, f"mutation site not unique: {old!r}"
    m = types.ModuleType("oracle_mutant")
    m.__package__ = "oracle"
    m.__file__ = SRC_PATH
    exec(compile(SRC.replace(old, new), SRC_PATH + " (mutant)", "exec"), m.__dict__)
    return m


def codecs_mutant(old, new):
    assert CODECS_SRC.count(old) == 1, f"mutation site not unique: {old!r}"
    m = types.ModuleType("codecs_mutant")
    m.__file__ = CODECS_PATH
    exec(compile(CODECS_SRC.replace(old, new), CODECS_PATH + " (mutant)", "exec"), m.__dict__)
    return m


def fails(pin, module=pins):
    name, args = (pin, ()) if isinstance(pin, str) else (pin[0], pin[1:])
    try:
        getattr(module, name)(*args)
    except Exception:
        return True
    return False


@pytest.mark.parametrize("slip,old,new,catchers", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_slip(monkeypatch, slip, old, new, catchers):
    monkeypatch.setattr(pins, "O", mutant(old, new))
    assert any(fails(p) for p in catchers), f"no pin caught: {slip}"


@pytest.mark.parametrize("slip,old,new,catchers", CODEC_MUTATIONS,
                         ids=[m[0] for m in CODEC_MUTATIONS])
def test_codec_pins_catch_planted_slip(monkeypatch, slip, old, new, catchers):
    monkeypatch.setattr(codec_pins, "codecs", codecs_mutant(old, new))
    assert any(fails(p, codec_pins) for p in catchers), f"no pin caught: {slip}"


def test_unmutated_oracle_passes_the_same_pins():
    """Control: every pin named above passes on the oracle as committed."""
    names = {p for m in MUTATIONS for p in m[3]}
    for p in sorted(names, key=str):
        assert not fails(p), p
    for p in sorted({p for m in CODEC_MUTATIONS for p in m[3]}):
        assert not fails(p, codec_pins), p
