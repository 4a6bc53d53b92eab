"""Pins of the oracle against what the Beam pages and the mathematics fix.

Each test checks the oracle against something other than itself: a value the pages print
(tests/golden/page_facts.json), a closed form, an invariant, a library routine (torch's
scaled_dot_product_attention, scipy's expit) or brute-force enumeration. Each is chosen so
that a plausible slip (a dropped term, a wrong sign or index, a transposed operand) fails.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle as O
from oracle.codecs import bf16_round, f32
from synth import BEAM, TINY

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")))


def rng(seed):
    return np.random.default_rng(seed)


# ------------------------------------------------------------------ residual stream ----

def test_rmsnorm_unit_rms_and_scale_invariance():
    x = rng(0).standard_normal((64, 512)) * 3.0
    y = O.rmsnorm(x, np.ones(512), 0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, atol=1e-12)
    assert np.allclose(O.rmsnorm(7.5 * x, np.ones(512), 0.0), y, atol=1e-12)
    w = rng(1).standard_normal(512)
    assert np.allclose(O.rmsnorm(x, w, 0.0), y * w, atol=1e-12)


@pytest.mark.parametrize("n", [2, 3, 5, 10, 52, 104, 105])
def test_depth_scaled_residual_keeps_unit_variance(n):
    """Beam page, MoE/residual section: with unit-variance sublayer outputs the n-th residual
    addition keeps the stream at unit variance. 10^6 samples; sampling error of the variance
    is ~0.14%, the bar is 0.5%. Writing h + x/sqrt(n) would give 1 + 1/n (>= 0.95% off)."""
    r = rng(n)
    H = 1000
    h = bf16_round(r.standard_normal((1000, H)))
    x = r.standard_normal((1000, H))
    h2, u = O.boundary_norm(x, h, np.ones(H), np.ones(H), n, 1e-6)
    assert abs(np.var(h2) - 1.0) < 5e-3
    # and the pre-norm of the new stream has unit RMS per row
    assert np.allclose(np.sqrt(np.mean(u * u, axis=-1)), 1.0, atol=4e-3)


def test_residual_first_term_and_coefficients():
    """n = 1 discards h entirely (sqrt(0) = 0): the stream becomes the normed sublayer output.
    The closed form with h = y pins the two coefficients: sqrt((n-1)/n) + 1/sqrt(n)."""
    H = 256
    x = rng(3).standard_normal((4, H))
    h = bf16_round(rng(4).standard_normal((4, H)))
    y = bf16_round(O.rmsnorm(x, np.ones(H), 1e-6))
    h1, _ = O.boundary_norm(x, h, np.ones(H), None, 1, 1e-6)
    assert np.array_equal(h1, y)
    for n in (2, 7, 104):
        hn, _ = O.boundary_norm(x, y, np.ones(H), None, n, 1e-6)
        c = math.sqrt((n - 1) / n) + 1 / math.sqrt(n)
        assert np.allclose(hn, y * c, rtol=2 ** -8, atol=0)


def test_first_boundary_is_pre_norm_only():
    H = 128
    e = bf16_round(rng(5).standard_normal((3, H)))
    w = 1 + 0.1 * rng(6).standard_normal(H)
    h, u = O.boundary_norm(None, e, None, w, 1, 1e-6)
    assert np.array_equal(h, e)
    assert np.allclose(u, bf16_round(O.rmsnorm(e, w, 1e-6)))


def test_layer_count_gives_104_boundaries():
    # two residual additions per layer after the embedding's n = 1
    L = GOLD["n_layers"]["value"]
    assert 2 * L == GOLD["residual_boundaries"]["value"]
    nope = [l for l in range(L) if O.is_nope_layer(l, L)]
    assert len(nope) == GOLD["kv_full_layers"]["value"]
    assert L - len(nope) == GOLD["n_swa_layers"]["value"]
    assert nope[-1] == L - 1 and nope[0] == 5


# ------------------------------------------------------------------ SSMax / RoPE ----

def test_ssmax_values():
    assert abs(O.ssmax_scale(1) - GOLD["ssmax_p1"]["value"]) < 1e-12
    assert abs(O.ssmax_scale(2048) - GOLD["ssmax_p2048"]["value"]) < 1e-12
    assert abs(O.ssmax_scale(2048) - 2 ** 0.1) < 1e-15


def test_rope_closed_forms():
    D, theta = 64, 10000.0
    for i in (0, 5, 31):
        e = np.zeros(D)
        e[i] = 1.0
        for m in (0, 1, 17, 4095):
            ang = m * theta ** (-2.0 * i / D)
            r = O.rope(e, m, theta)
            want = np.zeros(D)
            want[i] = math.cos(ang)
            want[i + D // 2] = math.sin(ang)
            assert np.allclose(r, want, atol=1e-12)


def test_rope_invariants():
    D, theta = 128, 10000.0
    r = rng(7)
    q, k = r.standard_normal(D), r.standard_normal(D)
    assert np.allclose(O.rope(q, 0, theta), q)
    assert abs(np.linalg.norm(O.rope(q, 12345, theta)) - np.linalg.norm(q)) < 1e-9
    d1 = O.rope(q, 100, theta) @ O.rope(k, 37, theta)
    d2 = O.rope(q, 100 + 5000, theta) @ O.rope(k, 37 + 5000, theta)
    assert abs(d1 - d2) < 1e-9


def _qkv_case(cfg, T, seed, nope, qn=None, kn=None):
    r = rng(seed)
    H, D = cfg.hidden, cfg.head_dim
    u = bf16_round(r.standard_normal((T, H)))
    w = bf16_round(0.02 * r.standard_normal((cfg.qkvg_rows, H)))
    qn = np.ones(D) if qn is None else qn
    kn = np.ones(D) if kn is None else kn
    cap = 64
    cache = O.KVCache(np.zeros((1, cfg.n_kv, cap, D)), np.zeros((1, cfg.n_kv, cap, D)),
                      window=0 if nope else cfg.window)
    return u, w, qn, kn, cache


def test_qkv_gate_nope_scales_q_only():
    """NoPE: |q'| per head = sqrt(D) * (1+p/2048)^0.1 with unit gains; k is not scaled."""
    cfg = TINY
    u, w, qn, kn, cache = _qkv_case(cfg, 2, 8, True)
    pos = np.array([1, 5000])          # scale 1.00005 and 1.131
    q, g = O.qkv_gate(cfg, u, w, qn, kn, [0, 0], pos, cache, nope=True)
    D = cfg.head_dim
    rms_q = np.sqrt(np.mean(q * q, axis=-1))                 # [T][Hq]
    for t, p in enumerate(pos):
        assert np.allclose(rms_q[t], O.ssmax_scale(p), rtol=3e-3)
    k = cache.k[0][:, cache.slot(pos), :]                     # [Hkv][T][D]
    assert np.allclose(np.sqrt(np.mean(k * k, axis=-1)), 1.0, rtol=3e-3)
    assert g.shape == (2, cfg.n_q * D)


def test_qkv_gate_packed_row_order():
    """The packed projection's rows are Q (Hq*D), K (Hkv*D), V (Hkv*D), gate (Hq*D), the order
    the Beam page lists them in (change 5). Each block of rows is filled with its own constant
    c_b, so with any u the projection of block b is c_b * sum(u): the cache's V holds the V
    block's value unnormalised and g the gate block's (a swapped pair of blocks fails)."""
    cfg = TINY
    Hq, Hkv, D = cfg.n_q, cfg.n_kv, cfg.head_dim
    sizes = [Hq * D, Hkv * D, Hkv * D, Hq * D]
    consts = [0.5, 0.25, 0.125, 0.0625]
    w = np.concatenate([np.full((n, cfg.hidden), c) for n, c in zip(sizes, consts)])
    u = np.full((1, cfg.hidden), 1.0 / cfg.hidden)          # sum(u) = 1
    cache = O.KVCache(np.zeros((1, Hkv, 8, D)), np.zeros((1, Hkv, 8, D)), window=cfg.window)
    q, g = O.qkv_gate(cfg, u, w, np.ones(D), np.ones(D), [0], [1], cache, nope=False)
    assert np.all(g == consts[3])
    assert np.all(cache.v[0, :, 0] == consts[2])
    assert np.allclose(cache.k[0, :, 0], 1.0, rtol=2 ** -8)   # a constant row, normed
    assert np.allclose(q, 1.0, rtol=2 ** -8)


def test_qkv_gate_rope_relative_position():
    """Sliding-window layer: q'.k depends only on the distance between the two positions."""
    cfg = TINY
    u, w, qn, kn, cache = _qkv_case(cfg, 2, 9, False)
    dots = []
    for shift in (0, 1000):
        pos = np.array([3, 9]) + shift
        c = O.KVCache(np.zeros_like(cache.k), np.zeros_like(cache.v), window=cfg.window)
        q, _ = O.qkv_gate(cfg, u, w, qn, kn, [0, 0], pos, c, nope=False)
        k0 = c.k[0][:, c.slot(pos[0]), :]                      # token 0's K, [Hkv][D]
        dots.append(np.einsum("hd,hd->h", q[1, ::cfg.n_q // cfg.n_kv], k0))
    assert np.allclose(dots[0], dots[1], rtol=2e-2, atol=2e-2)
    # position 1 is no rotation: q' is the plain normed q
    pos = np.array([1, 1])
    c = O.KVCache(np.zeros_like(cache.k), np.zeros_like(cache.v), window=cfg.window)
    q, _ = O.qkv_gate(cfg, u, w, qn, kn, [0, 0], pos, c, nope=False)
    z = bf16_round(u @ w.T)[:, : cfg.q_rows].reshape(2, cfg.n_q, cfg.head_dim)
    assert np.allclose(q, bf16_round(O.rmsnorm(z, qn, cfg.eps)))


# ------------------------------------------------------------------ KV cache size ----

def test_kv_cache_size_matches_page():
    vals = O.kv_values_per_token(GOLD["kv_full_layers"]["value"], BEAM.n_kv, BEAM.head_dim)
    assert vals == GOLD["kv_values_per_token"]["value"]
    assert vals * 2 == GOLD["kv_bytes_per_token_bf16"]["value"] == 36 * 1024
    assert vals * 1 == GOLD["kv_bytes_per_token_fp8"]["value"] == 18 * 1024
    assert vals * 1 * 2 ** 20 == GOLD["kv_bytes_1m_tokens_fp8_gib"]["value"] * 2 ** 30


def test_kv_cache_ring_and_fp8_roundtrip():
    D = 8
    k = np.zeros((1, 1, 4, D))
    c = O.KVCache(k, k.copy(), "bf16", window=4)
    for p in range(1, 8):
        c.store(0, p, np.full((1, D), p + 0.001), np.full((1, D), -p))
    kk, vv = c.load(0, np.arange(4, 8))
    assert np.allclose(kk[0, :, 0], bf16_round(np.arange(4, 8) + 0.001))
    assert np.array_equal(vv[0, :, 0], -np.arange(4, 8))
    # the layout the C ABI documents: 1-based position p lives in slot (p - 1) % capacity, so
    # positions 4..7 sit in slots 3, 0, 1, 2 of the raw array
    assert np.array_equal(c.v[0, 0, :, 0], [-5.0, -6.0, -7.0, -4.0])
    c8 = O.KVCache(np.zeros((1, 1, 4, D), np.uint8), np.zeros((1, 1, 4, D), np.uint8), "fp8",
                   k_scale=0.0371, v_scale=2.0)
    x = rng(10).standard_normal((1, D))
    c8.store(0, 2, x, x)
    kk, vv = c8.load(0, np.array([2]))
    # e4m3 keeps 3 fraction bits: relative error <= 2^-4 in the normal range
    assert np.allclose(kk[0, 0], x[0], rtol=2 ** -4, atol=0.0371 * 2 ** -9)
    assert np.allclose(vv[0, 0], x[0], rtol=2 ** -4, atol=2.0 * 2 ** -9)


# ------------------------------------------------------------------ attention ----

def _attn_setup(cfg, ctx, T, seed, window, cap=None):
    r = rng(seed)
    Hq, Hkv, D = cfg.n_q, cfg.n_kv, cfg.head_dim
    cap = cap or ctx + T
    k = bf16_round(r.standard_normal((1, Hkv, cap, D)))
    v = bf16_round(r.standard_normal((1, Hkv, cap, D)))
    cache = O.KVCache(k, v, window=window)
    q = bf16_round(r.standard_normal((T, Hq, D)))
    pos = np.arange(ctx + 1, ctx + T + 1)
    return cache, q, pos


def _attn_core(cfg, q, cache, pos):
    """Run the oracle's attention with the gate saturated to 1 and W_o = identity, so the
    output is bf16(o), the bare attention result."""
    T = q.shape[0]
    HD = cfg.n_q * cfg.head_dim
    g = np.full((T, HD), 200.0)
    return O.attention(cfg, q, g, np.zeros(cfg.n_q), cache, np.zeros(T, int), pos, np.eye(HD))


def test_attention_matches_torch_sdpa():
    """torch's scaled_dot_product_attention in float64 with an explicit band mask and KV
    heads repeated per query-head group (the library routine the definition reduces to)."""
    cfg = TINY
    ctx, T = 40, 6
    for window in (0, cfg.window):
        cache, q, pos = _attn_setup(cfg, ctx, T, 11, window)
        out = _attn_core(cfg, q, cache, pos)
        grp = cfg.n_q // cfg.n_kv
        kp = np.arange(1, ctx + T + 1)
        K = torch.from_numpy(cache.k[0][:, kp - 1]).repeat_interleave(grp, 0)   # [Hq][n][D]
        V = torch.from_numpy(cache.v[0][:, kp - 1]).repeat_interleave(grp, 0)
        Q = torch.from_numpy(q).permute(1, 0, 2)                              # [Hq][T][D]
        allow = kp[None, :] <= pos[:, None]
        if window:
            allow &= kp[None, :] > pos[:, None] - window
        mask = torch.from_numpy(allow)
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask)
        ref = bf16_round(ref.permute(1, 0, 2).reshape(T, -1).numpy())
        assert np.allclose(out, ref, rtol=2 ** -7, atol=1e-6)
        assert np.mean(out == ref) > 0.99


def test_attention_special_cases():
    cfg = TINY
    # a single key: the output is that key's value
    cache, q, pos = _attn_setup(cfg, 0, 1, 12, 0)
    out = _attn_core(cfg, q, cache, pos).reshape(cfg.n_q, cfg.head_dim)
    grp = cfg.n_q // cfg.n_kv
    for hq in range(cfg.n_q):
        assert np.array_equal(out[hq], cache.v[0, hq // grp, 0])
    # window >= context: sliding window equals full attention
    c1, q, pos = _attn_setup(cfg, 10, 3, 13, 0)
    c2 = O.KVCache(c1.k, c1.v, window=cfg.window)      # window 16 > 13 keys
    assert np.array_equal(_attn_core(cfg, q, c1, pos), _attn_core(cfg, q, c2, pos))
    # a ring buffer of capacity = window gives the same result as an unwrapped cache
    ctx = 50
    cbig, q, pos = _attn_setup(cfg, ctx, 1, 14, cfg.window)
    ring = O.KVCache(np.zeros((1, cfg.n_kv, cfg.window, cfg.head_dim)),
                     np.zeros((1, cfg.n_kv, cfg.window, cfg.head_dim)), window=cfg.window)
    for p in range(pos[0] - cfg.window + 1, pos[0] + 1):
        kk, vv = cbig.load(0, np.array([p]))
        ring.store(0, p, kk[:, 0], vv[:, 0])
    assert np.array_equal(_attn_core(cfg, q, cbig, pos), _attn_core(cfg, q, ring, pos))


def test_attention_gqa_head_mapping_and_gate():
    cfg = TINY
    cache, q, pos = _attn_setup(cfg, 5, 1, 15, 0)
    cache.v[0, 0] = 1.0
    cache.v[0, 1] = 2.0
    out = _attn_core(cfg, q, cache, pos).reshape(cfg.n_q, cfg.head_dim)
    grp = cfg.n_q // cfg.n_kv
    assert np.all(out[:grp] == 1.0) and np.all(out[grp:] == 2.0)
    # gate: g = 0, bias b -> output scaled by expit(b) per head
    HD = cfg.n_q * cfg.head_dim
    bias = np.array([-1.0, 0.0, 0.5, 3.0])
    out2 = O.attention(cfg, q, np.zeros((1, HD)), bias, cache, [0], pos, np.eye(HD))
    out2 = out2.reshape(cfg.n_q, cfg.head_dim)
    for hq in range(cfg.n_q):
        assert np.allclose(out2[hq], bf16_round(out[hq] * expit(bias[hq])))


# ------------------------------------------------------------------ router ----

def _route_case(cfg, T, seed):
    r = rng(seed)
    u = bf16_round(r.standard_normal((T, cfg.hidden)))
    wr = f32(0.02 * r.standard_normal((cfg.n_experts, cfg.hidden)))
    cb = f32(0.01 * r.standard_normal(cfg.n_experts))
    return u, wr, cb


def _brute_force_route(cfg, b):
    """Enumerate every choice of topk_groups groups (score: best pair of experts in each
    group), then every topk-subset of the kept groups' experts, maximising the total b."""
    E, G = b.shape[0], cfg.n_groups
    per = E // G
    def gscore(g):
        return max(b[i] + b[j] for i, j in itertools.combinations(range(g * per, (g + 1) * per), 2))
    gs = [gscore(g) for g in range(G)]
    best_groups = max(itertools.combinations(range(G), cfg.topk_groups),
                      key=lambda c: sum(gs[g] for g in c))
    cand = [e for g in best_groups for e in range(g * per, (g + 1) * per)]
    best = max(itertools.combinations(cand, cfg.topk), key=lambda c: sum(b[e] for e in c))
    return sorted(best)


def test_route_matches_brute_force_tiny():
    cfg = TINY
    u, wr, cb = _route_case(cfg, 64, 20)
    logits, s, b = O.route_scores(cfg, u, wr, cb)
    _, idx, w = O.route(cfg, u, wr, cb)
    for t in range(64):
        assert sorted(idx[t].tolist()) == _brute_force_route(cfg, b[t].astype(np.float64))
        assert abs(w[t].sum() - GOLD["route_scale"]["value"]) < 1e-5


def test_route_group_choice_full_width():
    """Beam width (8 groups of 32, top-4 groups, top-8): brute force over the 70 group
    choices, and every selected expert lies in a kept group and beats every unselected one
    there."""
    cfg = BEAM
    u, wr, cb = _route_case(cfg, 8, 21)
    _, s, b = O.route_scores(cfg, u, wr, cb)
    _, idx, w = O.route(cfg, u, wr, cb)
    per = cfg.n_experts // cfg.n_groups
    for t in range(8):
        bt = b[t].astype(np.float64)
        gs = [np.sort(bt[g * per:(g + 1) * per])[-2:].sum() for g in range(cfg.n_groups)]
        best = max(itertools.combinations(range(cfg.n_groups), cfg.topk_groups),
                   key=lambda c: sum(gs[g] for g in c))
        kept = [e for g in best for e in range(g * per, (g + 1) * per)]
        assert set(idx[t]) <= set(kept)
        rest = [e for e in kept if e not in set(idx[t])]
        assert bt[idx[t]].min() > bt[rest].max()
        assert list(bt[idx[t]]) == sorted(bt[idx[t]], reverse=True)


def test_route_weights_use_unbiased_scores():
    """The correction bias steers selection only: a large bias forces experts in, but their
    weights are their sigmoid scores, renormalised over the selection and scaled by 2.5."""
    cfg = TINY
    u, wr, cb = _route_case(cfg, 4, 22)
    cb = cb.copy()
    forced = [1, 2, 5, 6]                          # groups 0 and 1 hold experts 0-7
    cb[forced] = 10.0
    logits, idx, w = O.route(cfg, u, wr, cb)
    s = expit(logits.astype(np.float64))
    for t in range(4):
        assert sorted(idx[t].tolist()) == forced
        want = s[t, idx[t]] / s[t, idx[t]].sum() * 2.5
        assert np.allclose(w[t], want, rtol=1e-6)
    assert logits.dtype == np.float32


# ------------------------------------------------------------------ SwiGLU / MoE ----

def test_route_ties_go_to_lower_index():
    """READING (ties, not printed): equal scores rank by index, lower first, for groups and for
    experts. With every expert equal (identical router rows, zero bias) the first
    topk_groups groups are kept and the topk lowest experts of them chosen, in index order,
    each weighted route_scale / topk. Equal scores in one group only: the lower one wins."""
    cfg = TINY
    u = np.ones((1, cfg.hidden))
    wr = f32(np.full((cfg.n_experts, cfg.hidden), 0.01))
    cb = f32(np.zeros(cfg.n_experts))
    _, idx, w = O.route(cfg, u, wr, cb)
    assert idx[0].tolist() == list(range(cfg.topk))
    assert np.allclose(w, cfg.route_scale / cfg.topk)
    # experts 9 and 13 (groups 2 and 3) tie for the top score: both groups are kept and both
    # experts chosen, 9 listed first
    cb2 = cb.copy()
    cb2[[9, 13]] = 0.5
    _, idx2, _ = O.route(cfg, u, wr, cb2)
    assert idx2[0, 0] == 9 and idx2[0, 1] == 13


def test_route_gaps_match_subset_enumeration():
    """route_gaps against brute force: the group gap is the best total group score of any
    topk_groups-subset minus the second best (swapping the weakest kept group for the best
    dropped one), and the expert gap the same over the topk-subsets of the kept groups'
    experts. Ties planted in one token give a zero gap."""
    cfg = TINY
    u, wr, cb = _route_case(cfg, 24, 23)
    _, _, b = O.route_scores(cfg, u, wr, cb)
    b = b.astype(np.float64)
    per = cfg.n_experts // cfg.n_groups
    b[5] = np.tile(b[5, :per], cfg.n_groups)   # every group alike: tied group scores
    b[9] = 0.3                                 # every expert alike: tied everywhere
    gg, eg = O.route_gaps(cfg, b)
    for t in range(b.shape[0]):
        gs = [np.sort(b[t, g * per:(g + 1) * per])[-2:].sum() for g in range(cfg.n_groups)]
        tot = sorted((sum(gs[g] for g in c)
                      for c in itertools.combinations(range(cfg.n_groups), cfg.topk_groups)),
                     reverse=True)
        assert gg[t] == pytest.approx(tot[0] - tot[1], abs=1e-12)
        best = max(itertools.combinations(range(cfg.n_groups), cfg.topk_groups),
                   key=lambda c: (sum(gs[g] for g in c), [-g for g in c]))
        cand = [e for g in best for e in range(g * per, (g + 1) * per)]
        et = sorted((sum(b[t, e] for e in c) for c in itertools.combinations(cand, cfg.topk)),
                    reverse=True)
        assert eg[t] == pytest.approx(et[0] - et[1], abs=1e-12)
    assert gg[5] == 0.0 and eg[5] > 0.0
    assert gg[9] == 0.0 and eg[9] == 0.0


def test_route_gaps_bound_the_stable_perturbation():
    """Every biased score moved by less than min(group_gap/4, expert_gap/2) leaves the
    selection unchanged; a token whose gap is closed flips. Selection taken from route() via
    the correction bias (b = s + bias), with the sigmoid scores fixed."""
    cfg = TINY
    rng = np.random.default_rng(5)
    u, wr, cb = _route_case(cfg, 32, 24)
    logits, s, b = O.route_scores(cfg, u, wr, cb)
    _, idx0, _ = O.route(cfg, u, wr, cb)
    gg, eg = O.route_gaps(cfg, b)
    for t in range(32):
        lim = min(gg[t] / 4, eg[t] / 2)
        for _ in range(20):
            d = rng.uniform(-1, 1, cfg.n_experts) * lim * 0.9
            _, idx1, _ = O.route(cfg, u[t:t + 1], wr, f32(cb.astype(np.float64) + d))
            assert sorted(idx1[0]) == sorted(idx0[t])
    # close the expert gap of token 0: lift its best unselected kept-group expert past the
    # k-th selected one
    t = 0
    per = cfg.n_experts // cfg.n_groups
    groups = sorted({int(e) // per for e in idx0[t]})
    rest = [e for g in groups for e in range(g * per, (g + 1) * per) if e not in set(idx0[t])]
    e_in = int(idx0[t][-1])
    e_out = max(rest, key=lambda e: b[t, e])
    cb2 = cb.astype(np.float64).copy()
    cb2[e_out] += eg[t] * 1.5
    _, idx2, _ = O.route(cfg, u[t:t + 1], wr, f32(cb2))
    assert e_out in set(idx2[0]) and e_in not in set(idx2[0])


def test_silu_definition():
    z = np.linspace(-30, 30, 1001)
    assert np.allclose(O.silu(z), z * expit(z), rtol=1e-14, atol=1e-300)
    assert O.silu(np.array([0.0]))[0] == 0.0


def test_moe_equals_dense_with_stacked_experts():
    """With routing weights 1, the selected experts stacked into one dense SwiGLU of
    d_ff = k * F give the same output (Beam's dense d_ff 20480 = 8 x 2560)."""
    assert BEAM.d_ff_dense == BEAM.topk * BEAM.d_ff_expert
    cfg = TINY
    r = rng(23)
    H, F, E, k = cfg.hidden, cfg.d_ff_expert, cfg.n_experts, cfg.topk
    u = bf16_round(r.standard_normal((1, H)))
    wgu = bf16_round(0.02 * r.standard_normal((E, 2 * F, H)))
    wd = bf16_round(0.02 * r.standard_normal((E, H, F)))
    idx = np.array([[3, 9, 0, 14]])
    out = O.moe(cfg, u, idx, np.ones((1, k)), wgu, wd)
    gate = np.concatenate([wgu[e, :F] for e in idx[0]])
    up = np.concatenate([wgu[e, F:] for e in idx[0]])
    down = np.concatenate([wd[e] for e in idx[0]], axis=1)
    class Dense:
        d_ff_dense = k * F
    ref = O.dense_mlp(Dense, u, np.concatenate([gate, up]), down)
    assert np.allclose(out, ref, rtol=2 ** -7, atol=0)
    assert np.mean(out == ref) > 0.98


def test_moe_fp8_is_the_bf16_layer_on_dequantised_weights():
    """FP8 experts (weight-only): the layer on e4m3 codes times 128 x 128 block scales equals
    the BF16-weight layer on those values, decoded here by torch's float8_e4m3fn and expanded
    block by block with a Kronecker product (independent of the oracle's indexing)."""
    cfg = TINY
    H, F = cfg.hidden, cfg.d_ff_expert
    r = rng(31)

    def codes(rows, K):
        c = r.integers(0x20, 0x50, size=(rows, K), dtype=np.uint8)
        return (c | (r.integers(0, 2, size=(rows, K), dtype=np.uint8) << 7)).astype(np.uint8)

    def expand(sc, rows, K):
        return np.kron(sc.astype(np.float64), np.ones((128, 128)))[:rows, :K]

    def dec(c):
        return torch.from_numpy(c.copy()).view(torch.float8_e4m3fn).double().numpy()

    experts, gu, dn = {}, {}, {}
    for e in (1, 4, 6, 9):
        cg, cd = codes(2 * F, H), codes(H, F)
        sg = f32(r.uniform(0.002, 0.006, size=(-(-2 * F // 128), -(-H // 128))))
        sd = f32(r.uniform(0.002, 0.006, size=(-(-H // 128), -(-F // 128))))
        experts[e] = (cg, sg, cd, sd)
        gu[e] = dec(cg) * expand(sg, 2 * F, H)
        dn[e] = dec(cd) * expand(sd, H, F)
    u = bf16_round(r.standard_normal((3, H)))
    idx = np.array([[1, 4, 6, 9], [9, 6, 4, 1], [4, 1, 9, 6]])
    w = f32(r.uniform(0.1, 0.5, size=(3, 4))).astype(np.float64)
    assert np.array_equal(O.moe_fp8(cfg, u, idx, w, experts), O.moe(cfg, u, idx, w, gu, dn))


def test_moe_combine_is_weighted_sum():
    """Doubling one slot's weight adds exactly that expert's output once more."""
    cfg = TINY
    r = rng(24)
    H, F, E = cfg.hidden, cfg.d_ff_expert, cfg.n_experts
    u = bf16_round(r.standard_normal((1, H)))
    wgu = bf16_round(0.02 * r.standard_normal((E, 2 * F, H)))
    wd = bf16_round(0.02 * r.standard_normal((E, H, F)))
    one = O.moe(cfg, u, np.array([[5]]), np.ones((1, 1)), wgu, wd)
    two = O.moe(cfg, u, np.array([[5, 5]]), np.ones((1, 2)), wgu, wd)
    assert np.allclose(two, bf16_round(2 * one), rtol=2 ** -7)
    zero = O.moe(cfg, u, np.array([[5, 6]]), np.array([[1.0, 0.0]]), wgu, wd)
    assert np.array_equal(zero, one)


# ------------------------------------------------------------------ model size ----

def test_shapes_reproduce_page_parameter_counts():
    """Beam page: 501B parameters, 23B active. Non-embedding parameters of 52 layers (3 dense,
    49 MoE) at the stated widths must fall just under those (the vocabulary is not stated;
    ~1.3B embedding + LM head parameters close the gap)."""
    c = BEAM
    H = c.hidden
    attn = c.qkvg_rows * H + H * c.q_rows + 2 * c.head_dim + c.n_q + 4 * H
    dense = 3 * H * c.d_ff_dense
    expert = 3 * H * c.d_ff_expert
    router = c.n_experts * H + c.n_experts
    total = 52 * attn + 3 * dense + 49 * (c.n_experts * expert + router)
    active = 52 * attn + 3 * dense + 49 * (c.topk * expert + router)
    assert 498e9 < total < GOLD["total_params_b"]["value"] * 1e9
    assert 21e9 < active < GOLD["active_params_b"]["value"] * 1e9
    # the LM head's vocabulary reading: 201,088 rows (the vocabulary of the Harmony response
    # format the AREX feed article on the Day-0 support names), one matrix shared by the
    # embedding and the head, closes both gaps to the printed figures
    vocab = 201_088 * H
    assert round((total + vocab) / 1e9) == GOLD["total_params_b"]["value"]
    assert round((active + vocab) / 1e9) == GOLD["active_params_b"]["value"]


# ------------------------------------------------------------------ stack ----

def _tiny_stack(T_prefill, seed=0):
    cfg = TINY
    import synth
    Ws = []
    for l in range(cfg.n_layers):
        W = synth.layer_weights(cfg, l, seed)
        Ws.append({k: v.double().numpy() for k, v in W.items()})
    caches = []
    for l in range(cfg.n_layers):
        nope = O.is_nope_layer(l, cfg.n_layers)
        cap = 128
        z = np.zeros((1, cfg.n_kv, cap, cfg.head_dim))
        caches.append(O.KVCache(z, z.copy(), window=0 if nope else cfg.window))
    e = synth.activations(T_prefill, cfg.hidden, seed, "embed").double().numpy()
    return cfg, Ws, caches, e


def test_residual_index_counts_every_addition():
    """Beam page, MoE and residual-stream section and change 1: the n-th residual addition
    scales by sqrt((n-1)/n) and 1/sqrt(n), 104 of them for 52 layers after the embedding.
    Every boundary of a stack takes the next n: the embedding n = 1, then 2, 3, ..., 2L + 1,
    each once and in order (layer l's attention n = 2l + 2, its MLP n = 2l + 3)."""
    cfg, Ws, caches, e = _tiny_stack(1)
    g = O.stack_forward.__globals__          # the module whose boundary_norm the stack calls
    orig = g["boundary_norm"]
    seen = []

    def record(x, h, w_post, w_pre, n, eps):
        seen.append(n)
        return orig(x, h, w_post, w_pre, n, eps)

    g["boundary_norm"] = record
    try:
        O.stack_forward(cfg, Ws, caches, e, [0], [1])
    finally:
        g["boundary_norm"] = orig
    assert seen == list(range(1, 2 * cfg.n_layers + 2))


def test_stack_prefill_equals_token_by_token_decode():
    """Causality: a 20-token prefill gives the same per-token outputs as 20 single-token
    decode steps through the same caches (a mask that let a token see a later key, or a
    cache slot off by one, breaks it)."""
    cfg, Ws, caches, e = _tiny_stack(20)
    pos = np.arange(1, 21)
    h_all = O.stack_forward(cfg, Ws, caches, e, np.zeros(20, int), pos)
    cfg, Ws, caches2, _ = _tiny_stack(20)
    rows = [O.stack_forward(cfg, Ws, caches2, e[t:t + 1], [0], pos[t:t + 1]) for t in range(20)]
    ref = np.concatenate(rows)
    assert np.allclose(h_all, ref, rtol=2 ** -7, atol=0) and np.mean(h_all == ref) > 0.99
    rms = np.sqrt(np.mean(h_all ** 2, axis=-1))
    assert np.all((rms > 0.5) & (rms < 2.0))          # the depth-scaled stream stays O(1)


# ------------------------------------------------------------------------- LM head ----

def test_lm_head_softcap_closed_forms():
    """The page's cap c = 30 at closed-form points: tanh(ln 2) = 3/5 and tanh(ln 3) = 4/5 give
    18 and 24 at z = c ln 2 and c ln 3; the cap is odd, saturates at +-c, is the identity
    near 0 and keeps the order of the logits. A one-hot u makes z the first column of w_lm."""
    c = GOLD["logit_softcap"]["value"]
    zs = np.array([c * math.log(2), c * math.log(3), -c * math.log(2), 0.0, 1e-3, 1e4, -1e4])
    w = np.zeros((len(zs), 4))
    w[:, 0] = zs
    u = np.array([[1.0, 0.0, 0.0, 0.0]])
    got = O.lm_head(u, w, c)[0]
    want = [GOLD["softcap_at_30ln2"]["value"], GOLD["softcap_at_30ln3"]["value"],
            -GOLD["softcap_at_30ln2"]["value"], 0.0, 1e-3, c, -c]
    np.testing.assert_allclose(got, want, rtol=1e-6, atol=1e-9)
    z = rng(41).standard_normal(1000) * 40.0
    w = np.zeros((1000, 4))
    w[:, 0] = z
    y = O.lm_head(u, w, c)[0]
    assert np.all(np.abs(y) <= c)
    assert np.all(np.diff(y[np.argsort(z)]) >= 0)


def test_lm_head_projection_brute_force():
    """z[t][v] = sum_h u[t][h] w_lm[v][h] by explicit loops on small integers (exact), on a
    case with T, H and V all different, so a transposed operand cannot pass; softcap <= 0
    leaves z as it is."""
    r = rng(40)
    T, H, V = 3, 5, 7
    u = r.integers(-3, 4, (T, H)).astype(float)
    w = r.integers(-3, 4, (V, H)).astype(float)
    z = O.lm_head(u, w, 0.0)
    assert z.shape == (T, V)
    for t in range(T):
        for v in range(V):
            assert z[t, v] == sum(u[t, h] * w[v, h] for h in range(H))
