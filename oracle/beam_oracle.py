"""Oracle of one Beam decoder layer and of a truncated Beam stack (decode and prefill).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Sources. "Beam page" is the vLLM blog post "Reflection Beam 1.0 on vLLM: day-0 serving,
agent-optimised kernels, DFlash2 speculative decoding"; its sections used here are
  [Attn]  "Attention: sliding-window layers and NoPE full-attention layers"
  [MoE]   "MoE and residual stream: FP32 router, sandwich norm, depth-scaled residual"
  [Opt]   "Agent-driven optimisation speeds up batch-1 decode 2.71x" (the list of 7 changes)
  [Graph] "The fused decode graph runs one MoE layer in 13 kernels"
The stated choices where the pages are silent (RoPE theta 10000, group score = sum of the
two best biased scores, gate elementwise over the 6144-wide attention output, embedding =
residual term n=1) come with the task; every other reading is marked READING below.

Arithmetic: float64 throughout, with rounding to bfloat16 at each storage point and FP32
where the page fixes FP32 (the router). Values are passed as float64 arrays holding exactly
representable bf16/fp32 numbers; integer tensors as int arrays.
"""
from __future__ import annotations

import numpy as np

from .codecs import bf16_round, e4m3_decode, e4m3_encode, f32, fp8_block_dequant, nvfp4_dequant

__all__ = [
    "rmsnorm", "boundary_norm", "rope_inv_freq", "rope", "ssmax_scale", "KVCache",
    "qkv_gate", "attention", "route", "route_scores", "route_gaps", "silu", "moe", "moe_nvfp4",
    "moe_fp8", "dense_mlp",
    "is_nope_layer", "layer_forward", "stack_forward", "kv_values_per_token", "lm_head",
]


# ---------------------------------------------------------------------------------------
# RMSNorm and the boundary between sublayers  [MoE], [Opt] change 1
# ---------------------------------------------------------------------------------------

def rmsnorm(x, w, eps):
    """y = x / sqrt(mean(x^2) + eps) * w over the last axis.
    READING: plain gain w (not 1 + w); eps 1e-6 (not printed)."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)


def boundary_norm(x, h, w_post, w_pre, n, eps):
    """One sublayer boundary of the sandwich-norm residual stream [MoE]:

        y  = RMSNorm_post(x)                      (sublayer output, post-norm)
        h <- sqrt((n-1)/n) * h + y / sqrt(n)      (n-th residual addition)
        u  = RMSNorm_pre(h)                       (pre-norm of the next sublayer)

    x is None at the first boundary: h is then the embedding, residual term n = 1, and only
    the pre-norm runs. w_pre is None after the last sublayer. Storage points (READING of
    [Opt] change 1, "reference BF16 rounding points"): y, the new h and u are each rounded
    to bf16; everything between them is exact (float64)."""
    h = np.asarray(h, dtype=np.float64)
    if x is not None:
        y = bf16_round(rmsnorm(x, w_post, eps))
        h = bf16_round(np.sqrt((n - 1.0) / n) * h + y / np.sqrt(n))
    u = None if w_pre is None else bf16_round(rmsnorm(h, w_pre, eps))
    return h, u


# ---------------------------------------------------------------------------------------
# Positional treatment  [Attn]
# ---------------------------------------------------------------------------------------

def rope_inv_freq(D, theta):
    """Frequencies theta^(-2i/D), i = 0 .. D/2-1 (READING: rotary over the full head dim)."""
    i = np.arange(D // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / D)


def rope(x, m, theta):
    """Rotate x[..., D] by position index m (broadcast over x[..., 0]).
    READING: the half-split pairing (i, i + D/2), angle m * theta^(-2i/D); m = p - 1 for the
    1-based position p. cos/sin in float64."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    half = D // 2
    ang = np.asarray(m, dtype=np.float64)[..., None] * rope_inv_freq(D, theta)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def ssmax_scale(p, base=2048.0, expo=0.1):
    """SSMax query scale on NoPE layers: (1 + p/2048)^0.1 with 1-based position p [Attn]."""
    return np.power(1.0 + np.asarray(p, dtype=np.float64) / base, expo)


# ---------------------------------------------------------------------------------------
# KV cache  [Attn] (small KV cache), [Opt] change 6
# ---------------------------------------------------------------------------------------

class KVCache:
    """K and V of one layer, [S][Hkv][capacity][D]; position p lives in slot (p-1) % capacity.

    dtype "bf16": k, v hold float64 copies of bf16 values.
    dtype "fp8" : k, v hold uint8 e4m3 codes; value = code * scale, with one FP32 scale per
    tensor fixed when the cache is made (READING: per-layer per-tensor scales)."""

    def __init__(self, k, v, dtype="bf16", k_scale=1.0, v_scale=1.0, window=0):
        self.k = np.array(k)
        self.v = np.array(v)
        self.dtype = dtype
        self.k_scale = float(k_scale)
        self.v_scale = float(v_scale)
        self.window = int(window)      # 0: full context (NoPE), else sliding window W
        self.capacity = self.k.shape[2]

    def slot(self, p):
        return (np.asarray(p) - 1) % self.capacity

    def store(self, s, p, k_vec, v_vec):
        """Write one token's K and V ([Hkv][D], float64) at position p of sequence s."""
        sl = self.slot(p)
        if self.dtype == "fp8":
            # the quantisation decision is taken in FP32: code = e4m3(f32(x) / f32(scale))
            self.k[s, :, sl, :] = e4m3_encode(f32(k_vec) / np.float32(self.k_scale))
            self.v[s, :, sl, :] = e4m3_encode(f32(v_vec) / np.float32(self.v_scale))
        else:
            self.k[s, :, sl, :] = bf16_round(k_vec)
            self.v[s, :, sl, :] = bf16_round(v_vec)

    def load(self, s, positions):
        """K, V values [Hkv][len(positions)][D] (float64) of sequence s."""
        sl = self.slot(positions)
        k = self.k[s][:, sl, :]
        v = self.v[s][:, sl, :]
        if self.dtype == "fp8":
            return e4m3_decode(k) * self.k_scale, e4m3_decode(v) * self.v_scale
        return k.astype(np.float64), v.astype(np.float64)


def kv_values_per_token(n_full_layers, n_kv, head_dim):
    """Values a token leaves in the whole-sequence caches: layers x (K and V) x heads x dim."""
    return n_full_layers * 2 * n_kv * head_dim


# ---------------------------------------------------------------------------------------
# Packed QKV + gate projection, Q/K norm, RoPE or SSMax, cache write
#   [Attn], [Opt] changes 2, 5 and 6
# ---------------------------------------------------------------------------------------

def qkv_gate(cfg, u, w_qkvg, q_norm_w, k_norm_w, seq_id, pos, cache: KVCache, nope: bool):
    """Returns (q' [T][Hq][D], g [T][Hq*D]) and writes K, V of all T tokens into `cache`.

    Packed rows of w_qkvg, in order: Q (Hq*D), K (Hkv*D), V (Hkv*D), gate (Hq*D) [Opt] 5.
    q, k, v, g are rounded to bf16 as the projection's output (READING of the BF16 storage
    points). Per head, q and k are RMS-normalised over D with one shared [D] gain each
    (READING). Sliding-window layers then rotate q and k (RoPE); NoPE layers scale q by
    (1 + p/2048)^0.1 and leave k alone. q' is rounded to bf16; k, v go to the cache."""
    Hq, Hkv, D = cfg.n_q, cfg.n_kv, cfg.head_dim
    u = np.asarray(u, dtype=np.float64)
    T = u.shape[0]
    z = bf16_round(u @ np.asarray(w_qkvg, dtype=np.float64).T)
    q = z[:, : Hq * D].reshape(T, Hq, D)
    k = z[:, Hq * D: (Hq + Hkv) * D].reshape(T, Hkv, D)
    v = z[:, (Hq + Hkv) * D: (Hq + 2 * Hkv) * D].reshape(T, Hkv, D)
    g = z[:, (Hq + 2 * Hkv) * D:]
    qn = rmsnorm(q, q_norm_w, cfg.eps)
    kn = rmsnorm(k, k_norm_w, cfg.eps)
    pos = np.asarray(pos, dtype=np.int64)
    if nope:
        qn = qn * ssmax_scale(pos, cfg.ssmax_base, cfg.ssmax_exp)[:, None, None]
    else:
        m = (pos - 1)[:, None]
        qn = rope(qn, m, cfg.rope_theta)
        kn = rope(kn, m, cfg.rope_theta)
    for t in range(T):
        cache.store(int(seq_id[t]), int(pos[t]), kn[t], v[t])
    return bf16_round(qn), g


# ---------------------------------------------------------------------------------------
# Attention, output gate, o_proj  [Attn], [Opt] change 2
# ---------------------------------------------------------------------------------------

def attention(cfg, q, g, gate_bias, cache: KVCache, seq_id, pos, w_o):
    """GQA attention of each token over its sequence's cache, then the sigmoid gate and o_proj.

    Token at 1-based position p of sequence s attends to the keys at positions
    max(1, p-W+1) .. p on a sliding-window layer (READING: the 512-key window includes the
    token itself) and 1 .. p on a NoPE layer. Query head i uses KV head i // (Hq/Hkv)
    (READING). logits = q'.k / sqrt(D); softmax; o = P V, rounded to bf16. Then
    o <- o * sigmoid(g + bias[head]) (bias broadcast over the head's D columns), rounded to
    bf16, and out = o W_o^T rounded to bf16."""
    Hq, Hkv, D = cfg.n_q, cfg.n_kv, cfg.head_dim
    grp = Hq // Hkv
    q = np.asarray(q, dtype=np.float64)
    T = q.shape[0]
    o = np.zeros((T, Hq, D), dtype=np.float64)
    seq_id = np.asarray(seq_id, dtype=np.int64)
    pos = np.asarray(pos, dtype=np.int64)
    for s in np.unique(seq_id):
        toks = np.nonzero(seq_id == s)[0]
        pmax = int(pos[toks].max())
        lo_all = 1 if cache.window == 0 else max(1, int(pos[toks].min()) - cache.window + 1)
        kpos = np.arange(lo_all, pmax + 1)
        K, V = cache.load(int(s), kpos)          # [Hkv][nk][D]
        for t in toks:
            p = int(pos[t])
            lo = 1 if cache.window == 0 else max(1, p - cache.window + 1)
            a, b = lo - lo_all, p - lo_all + 1
            for hk in range(Hkv):
                qh = q[t, hk * grp:(hk + 1) * grp]                 # [grp][D]
                logits = qh @ K[hk, a:b].T / np.sqrt(D)           # [grp][nk]
                logits -= logits.max(axis=1, keepdims=True)
                e = np.exp(logits)
                o[t, hk * grp:(hk + 1) * grp] = (e / e.sum(axis=1, keepdims=True)) @ V[hk, a:b]
    o = bf16_round(o.reshape(T, Hq * D))
    gb = np.repeat(np.asarray(gate_bias, dtype=np.float64), D)
    gate = 1.0 / (1.0 + np.exp(-(np.asarray(g, dtype=np.float64) + gb)))
    og = bf16_round(o * gate)
    return bf16_round(og @ np.asarray(w_o, dtype=np.float64).T)


# ---------------------------------------------------------------------------------------
# Router  [MoE] (DeepSeek-V3 style, FP32)
# ---------------------------------------------------------------------------------------

def route_scores(cfg, u, w_router, corr_bias):
    """FP32 logits, sigmoid scores s and biased selection scores b = s + bias, each in FP32
    as the page requires (weights, accumulation and logits FP32; the accumulation here is
    float64, then rounded once)."""
    logits = f32(np.asarray(u, dtype=np.float64) @ np.asarray(w_router, dtype=np.float64).T)
    s = f32(1.0 / (1.0 + np.exp(-logits.astype(np.float64))))
    b = (s + f32(corr_bias)).astype(np.float32)          # FP32 addition
    return logits, s, b


def route(cfg, u, w_router, corr_bias):
    """Group-limited top-k routing. Returns (logits [T][E] fp32, idx [T][k], w [T][k]).

    Experts form n_groups contiguous groups (READING). Group score = sum of the two largest b
    in the group (stated choice), in FP32. Keep the topk_groups best groups, then the topk
    experts with the largest b among them; ties go to the lower index (READING). Weights use
    the unbiased s: w_j = s_j / sum(s_selected) * route_scale. idx is listed by descending b."""
    logits, s, b = route_scores(cfg, u, w_router, corr_bias)
    T, E = b.shape
    G = cfg.n_groups
    per = E // G
    idx = np.zeros((T, cfg.topk), dtype=np.int64)
    w = np.zeros((T, cfg.topk), dtype=np.float64)
    for t in range(T):
        bg = b[t].reshape(G, per)
        top2 = -np.sort(-bg, axis=1)[:, :2]
        gscore = (top2[:, 0] + top2[:, 1]).astype(np.float32)
        gorder = np.lexsort((np.arange(G), -gscore.astype(np.float64)))
        keep = gorder[: cfg.topk_groups]
        cand = np.concatenate([np.arange(g * per, (g + 1) * per) for g in np.sort(keep)])
        corder = np.lexsort((cand, -b[t, cand].astype(np.float64)))
        sel = cand[corder[: cfg.topk]]
        ssel = s[t, sel].astype(np.float64)
        idx[t] = sel
        w[t] = ssel / ssel.sum() * cfg.route_scale
    return logits, idx, f32(w)


def route_gaps(cfg, b):
    """How firmly each token's routing is decided, from its biased scores b [T][E].

    group_gap[t]  = group score of the last kept group minus that of the best dropped group
                    (the kG-th and (kG+1)-th largest group scores; inf when every group is kept)
    expert_gap[t] = the k-th largest biased score among the kept groups' experts minus the
                    (k+1)-th (inf when the kept groups hold exactly k experts)

    Group scores are the sums of the two largest b of each group, as in route(). If every b of
    a token moves by less than group_gap/4 (a group score then moves by less than group_gap/2)
    and by less than expert_gap/2, route() selects the same groups and the same experts; a gap
    of 0 is a tie that the index rule decides."""
    b = np.asarray(b, dtype=np.float64)
    T, E = b.shape
    G, kG, k = cfg.n_groups, cfg.topk_groups, cfg.topk
    per = E // G
    group_gap = np.full(T, np.inf)
    expert_gap = np.full(T, np.inf)
    for t in range(T):
        gscore = np.sort(b[t].reshape(G, per), axis=1)[:, -2:].sum(axis=1)
        order = np.lexsort((np.arange(G), -gscore))
        if kG < G:
            group_gap[t] = gscore[order[kG - 1]] - gscore[order[kG]]
        cand = np.sort(np.concatenate([b[t, g * per:(g + 1) * per] for g in order[:kG]]))[::-1]
        if k < cand.size:
            expert_gap[t] = cand[k - 1] - cand[k]
    return group_gap, expert_gap


# ---------------------------------------------------------------------------------------
# SwiGLU experts and dense MLP  [MoE], [Opt] changes 3 and 7
# ---------------------------------------------------------------------------------------

def silu(z):
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def _swiglu_act(u_t, w_gate_up, F):
    """a = silu(u W_gate^T) * (u W_up^T), rows of w_gate_up = [gate (F); up (F)] (READING),
    rounded to bf16 before the down projection."""
    gu = np.asarray(w_gate_up, dtype=np.float64) @ u_t
    return bf16_round(silu(gu[:F]) * gu[F:])


def moe(cfg, u, idx, w, w_gate_up, w_down):
    """out[t] = bf16( sum_j w[t,j] * y_tj ), y_tj = a_tj W_down[e]^T kept in FP32, summed in
    slot order j = 0..k-1 (READING). Only the selected experts are touched; w_gate_up and
    w_down may be arrays [E][..] or mappings expert -> array."""
    u = np.asarray(u, dtype=np.float64)
    T = u.shape[0]
    F = cfg.d_ff_expert
    out = np.zeros((T, u.shape[1]), dtype=np.float64)
    for t in range(T):
        acc = np.zeros(u.shape[1], dtype=np.float64)
        for j in range(idx.shape[1]):
            e = int(idx[t, j])
            a = _swiglu_act(u[t], w_gate_up[e], F)
            y = f32(np.asarray(w_down[e], dtype=np.float64) @ a).astype(np.float64)
            acc += float(w[t, j]) * y
        out[t] = acc
    return bf16_round(out)


def moe_nvfp4(cfg, u, idx, w, experts):
    """moe() with NVFP4 expert weights: experts maps expert e -> (gate_up codes [2F][H/2],
    gate_up block scales [2F][H/16], gate_up matrix scale, down codes [H][F/2], down block
    scales [H][F/16], down matrix scale). The selected experts' weights are dequantised
    exactly (every NVFP4 value is a float64 number) and the layer is the BF16-weight one."""
    used = sorted({int(e) for e in np.asarray(idx).ravel()})
    gu, dn = {}, {}
    for e in used:
        q_gu, s_gu, t_gu, q_dn, s_dn, t_dn = experts[e]
        gu[e] = nvfp4_dequant(q_gu, s_gu, t_gu)
        dn[e] = nvfp4_dequant(q_dn, s_dn, t_dn)
    return moe(cfg, u, idx, w, gu, dn)


def moe_fp8(cfg, u, idx, w, experts):
    """moe() with block-scaled FP8 expert weights (weight-only: the activations stay bf16):
    experts maps expert e -> (gate_up codes [2F][H], gate_up scales [2F/128][H/128], down codes
    [H][F], down scales [H/128][F/128]). The selected experts' weights are dequantised exactly
    and the layer is the BF16-weight one."""
    used = sorted({int(e) for e in np.asarray(idx).ravel()})
    gu, dn = {}, {}
    for e in used:
        c_gu, s_gu, c_dn, s_dn = experts[e]
        gu[e] = fp8_block_dequant(c_gu, s_gu)
        dn[e] = fp8_block_dequant(c_dn, s_dn)
    return moe(cfg, u, idx, w, gu, dn)


def dense_mlp(cfg, u, w_gate_up, w_down):
    """Dense SwiGLU of layers 0-2: bf16( a W_down^T ), a as in the experts, d_ff = d_ff_dense."""
    u = np.asarray(u, dtype=np.float64)
    Fd = cfg.d_ff_dense
    gu = u @ np.asarray(w_gate_up, dtype=np.float64).T
    a = bf16_round(silu(gu[:, :Fd]) * gu[:, Fd:])
    return bf16_round(a @ np.asarray(w_down, dtype=np.float64).T)


# ---------------------------------------------------------------------------------------
# Layer and stack  [Attn] (layer schedule), [MoE] (sandwich norm, residual index)
# ---------------------------------------------------------------------------------------

def is_nope_layer(layer, n_layers):
    """Full-attention NoPE layers are every 6th layer plus the last (READING: 0-based layer l
    is NoPE when (l + 1) % 6 == 0 or l is the last), giving 9 of Beam's 52 layers."""
    return (layer + 1) % 6 == 0 or layer == n_layers - 1


def layer_forward(cfg, l, W, h, u, cache, seq_id, pos, next_pre, trace=None):
    """Layer l of the stack, from (h, u = its attention pre-norm) to (h, u of the next layer).
    Residual terms (READING): the embedding is n = 1, layer l's attention is n = 2l+2 and its
    MLP n = 2l+3, so 52 layers give the page's 104 boundaries."""
    nope = is_nope_layer(l, cfg.n_layers)
    q, g = qkv_gate(cfg, u, W["w_qkvg"], W["q_norm"], W["k_norm"], seq_id, pos, cache, nope)
    a = attention(cfg, q, g, W["gate_bias"], cache, seq_id, pos, W["w_o"])
    h, u = boundary_norm(a, h, W["attn_post"], W["mlp_pre"], 2 * l + 2, cfg.eps)
    if l in cfg.dense_layers:
        m = dense_mlp(cfg, u, W["w_gate_up"], W["w_down"])
        r = None
    else:
        logits, idx, w = route(cfg, u, W["router"], W["corr_bias"])
        if "nvfp4_experts" in W:   # mapping expert -> its six NVFP4 arrays (moe_nvfp4)
            m = moe_nvfp4(cfg, u, idx, w, W["nvfp4_experts"])
        elif "fp8_experts" in W:   # mapping expert -> its four FP8 arrays (moe_fp8)
            m = moe_fp8(cfg, u, idx, w, W["fp8_experts"])
        else:
            m = moe(cfg, u, idx, w, W["w_gate_up"], W["w_down"])
        r = (logits, idx, w)
    if trace is not None:
        trace.append({"q": q, "g": g, "attn": a, "mlp_in": u, "mlp": m, "route": r})
    h, u = boundary_norm(m, h, W["mlp_post"], next_pre, 2 * l + 3, cfg.eps)
    return h, u


def stack_forward(cfg, weights, caches, e, seq_id, pos, trace=None):
    """Truncated stack over layers 0..L-1 for the tokens (seq_id, pos) with embeddings e.
    Returns h after the last residual addition (the final norm belongs to the LM head's
    input: boundary_norm(None, h, None, w_final, 1, eps)[1])."""
    h, u = boundary_norm(None, e, None, weights[0]["attn_pre"], 1, cfg.eps)
    L = cfg.n_layers
    for l in range(L):
        nxt = weights[l + 1]["attn_pre"] if l + 1 < L else None
        h, u = layer_forward(cfg, l, weights[l], h, u, caches[l], seq_id, pos, nxt, trace)
    return h


# ---------------------------------------------------------------------------------------
# LM head with the logit softcap  (AREX feed article on the Day-0 support, output side)
# ---------------------------------------------------------------------------------------

def lm_head(u, w_lm, softcap=30.0):
    """Logits of the final-normed hidden state u [T][H] over the vocabulary rows w_lm [V][H]:
    z = u w_lm^T, then logits = c * tanh(z / c) with c = softcap (30 on the page; c <= 0: no
    cap). Float64 math, FP32 result. READING: the head's input u is the final pre-norm
    RMSNorm_final(h) of the last residual stream, rounded to bf16 like every other pre-norm;
    the pages print neither the final norm nor the vocabulary size."""
    z = np.asarray(u, dtype=np.float64) @ np.asarray(w_lm, dtype=np.float64).T
    if softcap > 0:
        z = softcap * np.tanh(z / softcap)
    return f32(z)
