"""GPU parity, one C-ABI entry point at a time, against the oracle on the same seeded inputs.

Sizes: the tiny Beam-shaped widths (several tiles and ragged tails at small cost) and the
full Beam widths (hidden 5120, 48/8 heads of 128, 256 experts) at decode and prefill token
counts. Both sides get the same tensors; nothing the kernels produce is fed to the oracle.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
import synth
from synth import BEAM, TINY
from hybrid_attention_moe_gb300 import beam as B
from parity import (assert_close, assert_logits_close, codes_close, np64, oracle_cache,
                    route_margins)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def ws_for(cfg, T, max_pos=1):
    return torch.empty(B.workspace_bytes(cfg, T, max_pos), dtype=torch.uint8, device=DEV)


def cfg_of(shape, nope=False):
    return B.LayerCfg.from_shape(shape, B.BEAM_ATTN_NOPE_SSMAX if nope else B.BEAM_ATTN_SWA_ROPE)


def check_status():
    bits = B.beam_get_device_status()
    assert bits == 0, f"device status bits {bits:#x}"


# ------------------------------------------------------------------ boundary norm ----

@pytest.mark.parametrize("H,T", [(256, 1), (256, 37), (5120, 1), (5120, 8), (5120, 130)])
@pytest.mark.parametrize("n", [1, 2, 9, 104])
def test_boundary_norm(H, T, n):
    seed = 100 + n
    h = synth.activations(T, H, seed, "h")
    x = None if n == 1 else synth.activations(T, H, seed, "x")
    wpost = synth.normal((H,), 0.1, 1.0, seed, ("wpost",))
    wpre = synth.normal((H,), 0.1, 1.0, seed, ("wpre",))
    hd, ud = h.to(DEV), torch.empty_like(h, device=DEV)
    B.beam_boundary_norm(None if x is None else x.to(DEV), hd, ud,
                         None if x is None else wpost.to(DEV), wpre.to(DEV), n, 1e-6)
    h_ref, u_ref = O.boundary_norm(None if x is None else np64(x), np64(h), np64(wpost),
                                   np64(wpre), n, 1e-6)
    assert_close(np64(hd), h_ref, "h")
    assert_close(np64(ud), u_ref, "u")
    # last boundary: no next pre-norm
    if x is not None:
        hd2 = h.to(DEV)
        B.beam_boundary_norm(x.to(DEV), hd2, None, wpost.to(DEV), None, n, 1e-6)
        assert torch.equal(hd2, hd)


# ------------------------------------------------------------------ qkv + gate ----

def _qkv_inputs(shape, T, seed, positions, seqs, fp8, nope, scale=(1.0, 1.0)):
    W = synth.attention_weights(shape, 0, seed, device=DEV)
    u = synth.activations(T, shape.hidden, seed, "u", device=DEV)
    n_seqs = max(seqs) + 1
    if nope:
        cap = max(positions) + 8
        window = 0
    else:
        cap = shape.window + T + 3
        window = shape.window
    c = synth.kv_cache(shape, n_seqs, cap, seed, fp8=fp8, k_scale=scale[0], v_scale=scale[1],
                       device=DEV)
    kc = B.KVCache(c["k"], c["v"], window, scale[0], scale[1])
    seq = torch.tensor(seqs, dtype=torch.int32, device=DEV)
    pos = torch.tensor(positions, dtype=torch.int32, device=DEV)
    return W, u, kc, seq, pos


QKV_CASES = [
    # shape, T, positions, seqs
    (TINY, 1, [1], [0]),
    (TINY, 5, [3, 4, 5, 6, 7], [0, 0, 0, 0, 0]),
    (TINY, 40, list(range(90, 130)), [0] * 40),
    (BEAM, 1, [4097], [0]),
    (BEAM, 8, [100_001 + 977 * i for i in range(8)], list(range(8))),
    (BEAM, 48, list(range(2001, 2025)) + list(range(99_990, 100_014)), [0] * 24 + [1] * 24),
    (BEAM, 130, list(range(50_001, 50_131)), [0] * 130),          # tensor-core projection
]


@pytest.mark.parametrize("case", range(len(QKV_CASES)))
@pytest.mark.parametrize("nope", [False, True])
@pytest.mark.parametrize("fp8", [False, True])
def test_qkv_gate(case, nope, fp8):
    shape, T, positions, seqs = QKV_CASES[case]
    if nope:   # keep the whole-context cache small; RoPE keeps the large positions
        positions = [1 + p % 6000 for p in positions]
    scale = (0.0371, 0.5) if fp8 else (1.0, 1.0)
    W, u, kc, seq, pos = _qkv_inputs(shape, T, 7 + case, positions, seqs, fp8, nope, scale)
    cfg = cfg_of(shape, nope)
    oc = oracle_cache(kc)
    q = torch.empty((T, shape.n_q, shape.head_dim), dtype=torch.bfloat16, device=DEV)
    g = torch.empty((T, shape.q_rows), dtype=torch.bfloat16, device=DEV)
    B.beam_qkv_gate(cfg, u, W["w_qkvg"], W["q_norm"], W["k_norm"], seq, pos, q, g, kc,
                    ws_for(cfg, T))
    check_status()
    q_ref, g_ref = O.qkv_gate(shape, np64(u), np64(W["w_qkvg"]), np64(W["q_norm"]),
                              np64(W["k_norm"]), seqs, positions, oc, nope)
    assert_close(np64(q), q_ref, "q'")
    assert_close(np64(g), g_ref, "g")
    oc_gpu = oracle_cache(kc)
    for s, p in zip(seqs, positions):
        if fp8:
            sl = oc.slot(p)
            codes_close(oc_gpu.k[s][:, sl], oc.k[s][:, sl], kc.k_scale)
            codes_close(oc_gpu.v[s][:, sl], oc.v[s][:, sl], kc.v_scale)
        else:
            kg, vg = oc_gpu.load(s, np.array([p]))
            kr, vr = oc.load(s, np.array([p]))
            assert_close(kg, kr, "cached k")
            assert_close(vg, vr, "cached v")


# ------------------------------------------------------------------ attention ----

ATTN_CASES = [
    # shape, contexts (cached keys per sequence before the call), tokens per sequence
    (TINY, [0], 1),
    (TINY, [5, 40, 16, 3], 1),
    (TINY, [10], 64),            # prefill kernel, window boundary crossed mid-chunk
    (TINY, [30, 0], 40),         # two sequences in one prefill call
    (BEAM, [4096], 1),
    (BEAM, [300, 5000, 777, 12_345], 1),
    (BEAM, [2500], 48),
    (BEAM, [100, 700], 33),      # ragged prefill tile, two sequences
    (BEAM, [1000], 96),          # prefill kernel + tensor-core o_proj
]


# layer kind: NoPE (whole context), sliding window with the smallest ring, sliding window with
# the ring rounded up to a multiple of 128 slots (the layout the tensor-core prefill kernel
# takes for a ring)
ATTN_KINDS = ["nope", "swa", "swa_ring128"]


@pytest.mark.parametrize("case", range(len(ATTN_CASES)))
@pytest.mark.parametrize("kind", ATTN_KINDS)
@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("form", ["natural", "other"])
def test_attn(case, kind, fp8, form):
    """form 'natural' passes the true tokens per sequence (split-K decode up to 4, query tiles
    above: tensor-core tiles for a BF16 cache, else mma.sync tiles); 'other' forces the other
    form, which must give the same result. Cache slots past every query position hold NaN in
    NoPE layers: no kernel may let them reach a result."""
    nope = kind == "nope"
    shape, ctxs, per = ATTN_CASES[case]
    mq = per if form == "natural" else (64 if per <= 4 else 1)
    seed = 31 + case
    S = len(ctxs)
    T = S * per
    seqs = [s for s in range(S) for _ in range(per)]
    positions = [ctxs[s] + 1 + i for s in range(S) for i in range(per)]
    max_pos = max(positions)
    if nope:
        cap, window = max_pos + 5, 0
    else:
        cap, window = shape.window + per + 2, shape.window
        if kind == "swa_ring128":
            cap = -(-cap // 128) * 128
    scale = (0.0371, 0.5) if fp8 else (1.0, 1.0)
    c = synth.kv_cache(shape, S, cap, seed, fp8=fp8, k_scale=scale[0], v_scale=scale[1],
                       device=DEV)
    if nope:
        nan = 0x7F if fp8 else float("nan")     # e4m3fn code 0x7F is NaN
        c["k"][:, :, max_pos:] = nan
        c["v"][:, :, max_pos:] = nan
    kc = B.KVCache(c["k"], c["v"], window, *scale)
    q = synth.normal((T, shape.n_q, shape.head_dim), 1.0, 0.0, seed, ("q",), DEV)
    g = synth.activations(T, shape.q_rows, seed, "g", DEV)
    W = synth.attention_weights(shape, 0, seed, device=DEV)
    seq = torch.tensor(seqs, dtype=torch.int32, device=DEV)
    pos = torch.tensor(positions, dtype=torch.int32, device=DEV)
    cfg = cfg_of(shape, nope)
    out = torch.empty((T, shape.hidden), dtype=torch.bfloat16, device=DEV)
    B.beam_attn(cfg, q, g, W["gate_bias"], kc, seq, pos, max_pos, W["w_o"], out,
                ws_for(cfg, T, max_pos), max_q_per_seq=mq)
    check_status()
    ref = O.attention(shape, np64(q), np64(g), np64(W["gate_bias"]), oracle_cache(kc), seqs,
                      positions, np64(W["w_o"]))
    assert_close(np64(out), ref, "attn out", fp8=fp8)


@pytest.mark.parametrize("q_len", [2, 4, 7, 8])
@pytest.mark.parametrize("kind", ["nope", "swa_ring128"])
@pytest.mark.parametrize("form", ["decode", "grouped", "prefill"])
def test_attn_verify_batches(q_len, kind, form):
    """Multi-token verification batches of speculative decoding at full width: q_len new tokens
    per sequence (2 sequences) after 100,000 cached ones, through every form of beam_attn --
    split-K decode per token (which a bound of 1 always takes), the grouped form in which a
    sequence's tokens share each K/V block (the true bound, full attention over a BF16 cache)
    and the query-tile prefill kernel (a bound above 16) -- whatever q_len is."""
    shape = BEAM
    nope = kind == "nope"
    if form == "grouped" and not nope:
        pytest.skip("a 512-key window takes the per-token decode kernels whatever the bound")
    ctxs = [100_000, 99_123]
    S = len(ctxs)
    T = S * q_len
    seed = 300 + q_len
    seqs = [s for s in range(S) for _ in range(q_len)]
    positions = [ctxs[s] + 1 + i for s in range(S) for i in range(q_len)]
    max_pos = max(positions)
    cap, window = (max_pos + 5, 0) if nope else (-(-(shape.window + q_len + 2) // 128) * 128,
                                                  shape.window)
    c = synth.kv_cache(shape, S, cap, seed, device=DEV)
    kc = B.KVCache(c["k"], c["v"], window)
    q = synth.normal((T, shape.n_q, shape.head_dim), 1.0, 0.0, seed, ("q",), DEV)
    g = synth.activations(T, shape.q_rows, seed, "g", DEV)
    W = synth.attention_weights(shape, 0, seed, device=DEV)
    seq = torch.tensor(seqs, dtype=torch.int32, device=DEV)
    pos = torch.tensor(positions, dtype=torch.int32, device=DEV)
    cfg = cfg_of(shape, nope)
    out = torch.empty((T, shape.hidden), dtype=torch.bfloat16, device=DEV)
    # a bound above 16 always takes the query tiles
    mq = {"decode": 1, "grouped": q_len, "prefill": 17}[form]
    B.beam_attn(cfg, q, g, W["gate_bias"], kc, seq, pos, max_pos, W["w_o"], out,
                ws_for(cfg, T, max_pos), max_q_per_seq=mq)
    check_status()
    ref = O.attention(shape, np64(q), np64(g), np64(W["gate_bias"]), oracle_cache(kc), seqs,
                      positions, np64(W["w_o"]))
    assert_close(np64(out), ref, "attn out")


# The grouped verification form over layouts a serving batch can take: runs of different
# lengths (one of a single token), a sequence's tokens interleaved with other sequences' (they
# still share blocks only where consecutive), many short groups at 8K context (pairs whole in
# one CTA and pairs split between CTAs), 16 tokens of one sequence (96 query columns, the
# widest group) and runs longer than the bound (split into groups of the bound). Every slot past
# a sequence's last position holds NaN, so keys a column must not see cannot leak.
GROUPED_CASES = {
    # name: (tokens as (sequence, position) in call order, contexts per sequence, bound)
    "runs": ([(0, 3001 + i) for i in range(5)] + [(1, 2501)] + [(2, 4101 + i) for i in range(9)],
             [3000, 2500, 4100], 9),
    "interleaved": ([(0, 2201), (1, 3301), (0, 2202), (1, 3302), (2, 2801), (0, 2203), (2, 2802)],
                    [2200, 3300, 2800], 3),
    "many": ([(s, 2100 + 397 * s + 1 + i) for s in range(16) for i in range(2)],
             [2100 + 397 * s for s in range(16)], 2),
    "q16": ([(0, 100_001 + i) for i in range(16)], [100_000], 16),
    "split_runs": ([(s, 5000 + 77 * s + 1 + i) for s in range(2) for i in range(8)],
                   [5000, 5077], 4),
}


@pytest.mark.parametrize("name", list(GROUPED_CASES))
def test_attn_grouped_layouts(name):
    shape = BEAM
    tokens, ctxs, mq = GROUPED_CASES[name]
    seqs = [s for s, _ in tokens]
    positions = [p for _, p in tokens]
    S, T = len(ctxs), len(tokens)
    max_pos = max(positions)
    cap = max_pos + 7
    seed = 900 + T
    c = synth.kv_cache(shape, S, cap, seed, device=DEV)
    for s in range(S):
        last = max(p for t, p in tokens if t == s)
        c["k"][s, :, last:] = float("nan")
        c["v"][s, :, last:] = float("nan")
    kc = B.KVCache(c["k"], c["v"], 0)
    q = synth.normal((T, shape.n_q, shape.head_dim), 1.0, 0.0, seed, ("q",), DEV)
    g = synth.activations(T, shape.q_rows, seed, "g", DEV)
    W = synth.attention_weights(shape, 0, seed, device=DEV)
    seq = torch.tensor(seqs, dtype=torch.int32, device=DEV)
    pos = torch.tensor(positions, dtype=torch.int32, device=DEV)
    cfg = cfg_of(shape, nope=True)
    out = torch.empty((T, shape.hidden), dtype=torch.bfloat16, device=DEV)
    B.beam_attn(cfg, q, g, W["gate_bias"], kc, seq, pos, max_pos, W["w_o"], out,
                ws_for(cfg, T, max_pos), max_q_per_seq=mq)
    check_status()
    ref = O.attention(shape, np64(q), np64(g), np64(W["gate_bias"]), oracle_cache(kc), seqs,
                      positions, np64(W["w_o"]))
    assert_close(np64(out), ref, f"attn out ({name})")


@pytest.mark.parametrize("bad", ["position", "sequence"])
def test_grouped_form_flags_bad_tokens(bad):
    """Grouped form: a token whose position lies past the host's max_pos (its group's other
    tokens still exact), or a group whose sequence id is out of range: the status word says so
    and the bad rows are left at zero; the other tokens are exact."""
    shape = BEAM
    cfg = cfg_of(shape, nope=True)
    cap, max_pos = 5000, 3000
    c = synth.kv_cache(shape, 1, cap, 5, device=DEV)
    kc = B.KVCache(c["k"], c["v"], 0)
    if bad == "position":
        seqs, positions = [0, 0, 0], [2500, 2501, 4000]
    else:
        seqs, positions = [0, 0, 3], [2500, 2501, 2900]
    T = len(seqs)
    q = synth.normal((T, shape.n_q, shape.head_dim), 1.0, 0.0, 5, ("q",), DEV)
    g = synth.activations(T, shape.q_rows, 5, "g", DEV)
    W = synth.attention_weights(shape, 0, 5, device=DEV)
    out = torch.empty((T, shape.hidden), dtype=torch.bfloat16, device=DEV)
    B.beam_get_device_status()
    B.beam_attn(cfg, q, g, W["gate_bias"], kc, torch.tensor(seqs, dtype=torch.int32, device=DEV),
                torch.tensor(positions, dtype=torch.int32, device=DEV), max_pos, W["w_o"], out,
                ws_for(cfg, T, max_pos), max_q_per_seq=3)
    assert B.beam_get_device_status() & (B.DEV_BAD_POSITION if bad == "position"
                                         else B.DEV_BAD_SEQ)
    ref = O.attention(shape, np64(q[:2]), np64(g[:2]), np64(W["gate_bias"]), oracle_cache(kc),
                      seqs[:2], positions[:2], np64(W["w_o"]))
    assert_close(np64(out[:2]), ref, "attn out, valid tokens")
    assert not out[2].float().abs().max().item()


# A sliding window longer than 2048 keys takes the long-context decode kernel when the ring's
# capacity is a multiple of its key block (64 slots for BF16, 128 for FP8) and the split-K kernel
# otherwise; the contexts make the window wrap around the ring and one sequence hold fewer
# keys than the window.
LONG_WINDOW = dataclasses.replace(BEAM, window=3000)


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("cap", [3072, 3136, 3005])
@pytest.mark.parametrize("per", [1, 3])
def test_attn_long_window_ring(fp8, cap, per):
    shape = LONG_WINDOW
    seed = 71 + cap + per
    ctxs = [5000, 2999, 7000, 12]
    S = len(ctxs)
    T = S * per
    seqs = [s for s in range(S) for _ in range(per)]
    positions = [ctxs[s] + 1 + i for s in range(S) for i in range(per)]
    max_pos = max(positions)
    scale = (0.0371, 0.5) if fp8 else (1.0, 1.0)
    c = synth.kv_cache(shape, S, cap, seed, fp8=fp8, k_scale=scale[0], v_scale=scale[1],
                       device=DEV)
    kc = B.KVCache(c["k"], c["v"], shape.window, *scale)
    q = synth.normal((T, shape.n_q, shape.head_dim), 1.0, 0.0, seed, ("q",), DEV)
    g = synth.activations(T, shape.q_rows, seed, "g", DEV)
    W = synth.attention_weights(shape, 0, seed, device=DEV)
    seq = torch.tensor(seqs, dtype=torch.int32, device=DEV)
    pos = torch.tensor(positions, dtype=torch.int32, device=DEV)
    cfg = cfg_of(shape)
    out = torch.empty((T, shape.hidden), dtype=torch.bfloat16, device=DEV)
    B.beam_attn(cfg, q, g, W["gate_bias"], kc, seq, pos, max_pos, W["w_o"], out,
                ws_for(cfg, T, max_pos), max_q_per_seq=per)
    check_status()
    ref = O.attention(shape, np64(q), np64(g), np64(W["gate_bias"]), oracle_cache(kc), seqs,
                      positions, np64(W["w_o"]))
    assert_close(np64(out), ref, "attn out", fp8=fp8)


def test_long_context_decode_flags_positions_past_max_pos():
    """The long-context decode kernel sizes its key blocks from max_pos: a token whose position
    lies past it is flagged and its row left at zero, the other tokens are exact."""
    shape = BEAM
    cfg = cfg_of(shape, nope=True)
    S, cap, max_pos = 2, 5000, 3000
    c = synth.kv_cache(shape, S, cap, 3, device=DEV)
    kc = B.KVCache(c["k"], c["v"], 0)
    seqs, positions = [0, 1], [2500, 4000]
    q = synth.normal((S, shape.n_q, shape.head_dim), 1.0, 0.0, 3, ("q",), DEV)
    g = synth.activations(S, shape.q_rows, 3, "g", DEV)
    W = synth.attention_weights(shape, 0, 3, device=DEV)
    out = torch.empty((S, shape.hidden), dtype=torch.bfloat16, device=DEV)
    B.beam_get_device_status()
    B.beam_attn(cfg, q, g, W["gate_bias"], kc, torch.tensor(seqs, dtype=torch.int32, device=DEV),
                torch.tensor(positions, dtype=torch.int32, device=DEV), max_pos, W["w_o"], out,
                ws_for(cfg, S, max_pos), max_q_per_seq=1)
    assert B.beam_get_device_status() & B.DEV_BAD_POSITION
    ref = O.attention(shape, np64(q[:1]), np64(g[:1]), np64(W["gate_bias"]), oracle_cache(kc),
                      seqs[:1], positions[:1], np64(W["w_o"]))
    assert_close(np64(out[:1]), ref, "attn out, valid token")
    assert not out[1].float().abs().max().item()


# ------------------------------------------------------------------ router ----

# Router shapes beside the Beam and tiny ones: 96 experts in 3 groups of 32 (4 experts per lane,
# a group spanning 8 lanes of the warp-per-token top-k) and 48 experts in 4 groups of 12 (a group
# not a power-of-two number of lanes: the CTA-per-token top-k).
ROUTE_96 = dataclasses.replace(TINY, n_experts=96, n_groups=3, topk_groups=2, topk=6)
ROUTE_48 = dataclasses.replace(TINY, n_experts=48, n_groups=4, topk_groups=2, topk=4)


@pytest.mark.parametrize("shape,T", [(TINY, 1), (TINY, 77), (BEAM, 1), (BEAM, 8), (BEAM, 300),
                                     (ROUTE_96, 5), (ROUTE_48, 1), (ROUTE_48, 40),
                                     (TINY, 700), (BEAM, 1030)])
def test_route(shape, T):
    """FP32 SIMT logits below 512 tokens; from 512 the tensor-core GEMM over the exact
    three-part BF16 split of the FP32 router weights (same logits to FP32 rounding)."""
    cfg = cfg_of(shape)
    for attempt in range(20):
        seed = 1000 * attempt + T
        u = synth.activations(T, shape.hidden, seed, "u")
        R = synth.router_weights(shape, 0, seed)
        gmin, emin = route_margins(shape, np64(u), np64(R["router"]), np64(R["corr_bias"]))
        if min(gmin, emin) >= 1e-6:
            break
    else:
        pytest.fail("no tie-free draw")
    logits = torch.empty((T, shape.n_experts), dtype=torch.float32, device=DEV)
    idx = torch.empty((T, shape.topk), dtype=torch.int32, device=DEV)
    w = torch.empty((T, shape.topk), dtype=torch.float32, device=DEV)
    B.beam_route(cfg, u.to(DEV), R["router"].to(DEV), R["corr_bias"].to(DEV), logits, idx, w,
                 ws_for(cfg, T))
    lg_ref, idx_ref, w_ref = O.route(shape, np64(u), np64(R["router"]), np64(R["corr_bias"]))
    assert_logits_close(logits.cpu().double().numpy(), lg_ref)
    gi, gw = idx.cpu().numpy(), w.cpu().double().numpy()
    for t in range(T):
        assert sorted(gi[t].tolist()) == sorted(idx_ref[t].tolist()), f"token {t}"
        assert gi[t].tolist() == idx_ref[t].tolist()     # gaps >= 1e-6 fix the order too
    assert np.max(np.abs(gw - w_ref) / np.abs(w_ref)) < 1e-5
    # no logits buffer: selection identical
    idx2 = torch.empty_like(idx)
    w2 = torch.empty_like(w)
    B.beam_route(cfg, u.to(DEV), R["router"].to(DEV), R["corr_bias"].to(DEV), None, idx2, w2,
                 ws_for(cfg, T))
    assert torch.equal(idx2, idx) and torch.equal(w2, w)


# ------------------------------------------------------------------ experts ----

def _random_routing(shape, T, seed, n_used=None):
    rng = np.random.default_rng(seed)
    pool = np.arange(shape.n_experts) if n_used is None else \
        rng.choice(shape.n_experts, n_used, replace=False)
    idx = np.stack([rng.choice(pool, shape.topk, replace=False) for _ in range(T)])
    w = rng.uniform(0.05, 0.6, size=(T, shape.topk)).astype(np.float32)
    return idx.astype(np.int32), w


@pytest.mark.parametrize("shape,T,n_used", [(TINY, 1, None), (TINY, 3, 5), (TINY, 4, None),
                                            (TINY, 9, None), (TINY, 31, None), (TINY, 32, None),
                                            (TINY, 300, None), (BEAM, 1, None), (BEAM, 2, None),
                                            (BEAM, 4, None), (BEAM, 8, None), (BEAM, 40, 12),
                                            (BEAM, 200, 10)])
def test_moe(shape, T, n_used):
    """One token: its slots used directly by the SIMT weight-streaming kernels; 2 to 31 tokens:
    mma.sync expert products after the plan (up to 8 pairs of an expert per pass over its
    rows; T=31 on the tiny shape gives experts more than 8 pairs), the down kernel's last CTA
    per row block combines; grouped tensor-core GEMMs from 32 tokens (n_used limits the
    distinct experts so several 128-row tiles and ragged tails occur per expert)."""
    seed = 55 + T
    cfg = cfg_of(shape)
    idx, w = _random_routing(shape, T, seed, n_used)
    if shape is TINY:
        wgu, wdn = synth.expert_weights(shape, 0, seed, device=DEV)
    else:   # only the experts used, placed at their indices of a full-size tensor
        E, F, H = shape.n_experts, shape.d_ff_expert, shape.hidden
        wgu = torch.zeros((E, 2 * F, H), dtype=torch.bfloat16, device=DEV)
        wdn = torch.zeros((E, H, F), dtype=torch.bfloat16, device=DEV)
        used = sorted(set(idx.ravel().tolist()))
        gu, dn = synth.expert_weights(shape, 0, seed, device=DEV, experts=used)
        for i, e in enumerate(used):
            wgu[e], wdn[e] = gu[i], dn[i]
    u = synth.activations(T, shape.hidden, seed, "u", DEV)
    out = torch.empty((T, shape.hidden), dtype=torch.bfloat16, device=DEV)
    B.beam_moe(cfg, u, torch.from_numpy(idx).to(DEV), torch.from_numpy(w).to(DEV), wgu, wdn,
               out, ws_for(cfg, T))
    check_status()
    used = sorted(set(idx.ravel().tolist()))
    ogu = {e: np64(wgu[e]) for e in used}
    odn = {e: np64(wdn[e]) for e in used}
    ref = O.moe(shape, np64(u), idx, w.astype(np.float64), ogu, odn)
    assert_close(np64(out), ref, "moe out")


@pytest.mark.parametrize("shape", [TINY, BEAM])
def test_moe_bad_expert_slots_flagged_and_skipped(shape):
    """One token with two slots naming experts out of range: the status word says so and the
    output is the combine of the valid slots only (full width: the balanced one-token kernels;
    tiny: the row-per-warp ones)."""
    cfg = cfg_of(shape)
    E, F, H, k = shape.n_experts, shape.d_ff_expert, shape.hidden, shape.topk
    valid = list(range(k - 2))
    row = valid[:1] + [E + 5] + valid[1:] + [-2]
    idx = np.asarray([row], dtype=np.int32)
    w = np.linspace(0.1, 0.5, k, dtype=np.float32)[None, :]
    wgu = torch.zeros((E, 2 * F, H), dtype=torch.bfloat16, device=DEV)
    wdn = torch.zeros((E, H, F), dtype=torch.bfloat16, device=DEV)
    gu, dn = synth.expert_weights(shape, 0, 7, device=DEV, experts=valid)
    for i, e in enumerate(valid):
        wgu[e], wdn[e] = gu[i], dn[i]
    u = synth.activations(1, H, 7, "u", DEV)
    out = torch.empty((1, H), dtype=torch.bfloat16, device=DEV)
    B.beam_get_device_status()
    B.beam_moe(cfg, u, torch.from_numpy(idx).to(DEV), torch.from_numpy(w).to(DEV), wgu, wdn,
               out, ws_for(cfg, 1))
    assert B.beam_get_device_status() & B.DEV_BAD_EXPERT
    keep = [j for j in range(k) if 0 <= row[j] < E]
    ref = O.moe(shape, np64(u), idx[:, keep], w[:, keep].astype(np.float64),
                {e: np64(wgu[e]) for e in valid}, {e: np64(wdn[e]) for e in valid})
    assert_close(np64(out), ref, "moe out, valid slots")


def _nvfp4_experts(shape, used, seed):
    """NVFP4 expert tensors on the device (only the used experts drawn, the rest zero) and
    the oracle's view of the used ones."""
    E, F, H = shape.n_experts, shape.d_ff_expert, shape.hidden
    part = synth.expert_weights_nvfp4(shape, 0, seed, device=DEV, experts=used)
    full = {
        "gate_up": torch.zeros((E, 2 * F, H // 2), dtype=torch.uint8, device=DEV),
        "gate_up_scale": torch.zeros((E, 2 * F, H // 16), dtype=torch.uint8, device=DEV),
        "gate_up_global": torch.zeros((E,), dtype=torch.float32, device=DEV),
        "down": torch.zeros((E, H, F // 2), dtype=torch.uint8, device=DEV),
        "down_scale": torch.zeros((E, H, F // 16), dtype=torch.uint8, device=DEV),
        "down_global": torch.zeros((E,), dtype=torch.float32, device=DEV),
    }
    for i, e in enumerate(used):
        for k in full:
            full[k][e] = part[k][i]
    host = {k: v.cpu().numpy() for k, v in part.items()}
    experts = {e: (host["gate_up"][i], host["gate_up_scale"][i], host["gate_up_global"][i],
                   host["down"][i], host["down_scale"][i], host["down_global"][i])
               for i, e in enumerate(used)}
    return full, experts


# a second small shape (hidden and d_ff multiples of 256, 4 of 16 experts per token), and one
# with 64 experts, 8 per token: from 32 tokens its active experts span several dequantisation
# chunks of the grouped GEMM path
NVFP4_MID = dataclasses.replace(TINY, hidden=512, d_ff_expert=256)
NVFP4_WIDE = dataclasses.replace(TINY, hidden=512, d_ff_expert=256, n_experts=64, n_groups=8,
                                 topk_groups=4, topk=8)


@pytest.mark.parametrize("shape,T,n_used", [(TINY, 1, None), (TINY, 3, 5), (TINY, 5, None),
                                            (TINY, 13, None), (TINY, 31, 6), (NVFP4_MID, 1, None),
                                            (NVFP4_MID, 2, None), (BEAM, 1, None),
                                            (BEAM, 2, None), (BEAM, 4, None), (BEAM, 8, None),
                                            (TINY, 32, None), (TINY, 300, None),
                                            (NVFP4_MID, 64, 5), (NVFP4_WIDE, 64, None),
                                            (NVFP4_WIDE, 130, 37), (BEAM, 48, 9)])
def test_moe_nvfp4(shape, T, n_used):
    """NVFP4 expert weights (e2m1 codes, e4m3 block scales, FP32 matrix scales): below 32
    tokens mma.sync f16 products of the dequantised weights, the selected experts only; up to 4
    tokens four warps split each row block's K (T=4 and T=5 sit on either side); T=31 over 6
    experts gives experts more than 8 pairs (several passes). From 32 tokens the grouped BF16
    tensor-core GEMMs on weights dequantised chunk by chunk (NVFP4_WIDE at 130 tokens over 37
    experts: three chunks)."""
    seed = 91 + T
    cfg = cfg_of(shape)
    idx, w = _random_routing(shape, T, seed, n_used)
    used = sorted(set(idx.ravel().tolist()))
    full, experts = _nvfp4_experts(shape, used, seed)
    u = synth.activations(T, shape.hidden, seed, "u", DEV)
    out = torch.empty((T, shape.hidden), dtype=torch.bfloat16, device=DEV)
    B.beam_moe_nvfp4(cfg, u, torch.from_numpy(idx).to(DEV), torch.from_numpy(w).to(DEV), full,
                     out, ws_for(cfg, T))
    check_status()
    ref = O.moe_nvfp4(shape, np64(u), idx, w.astype(np.float64), experts)
    assert_close(np64(out), ref, "moe nvfp4 out")


@pytest.mark.parametrize("shape", [TINY, NVFP4_MID])
def test_moe_nvfp4_bad_expert_slots_flagged_and_skipped(shape):
    cfg = cfg_of(shape)
    for rows in ([[0, 1, 99, 2]], [[0, 1, 99, 2], [5, -3, 1, 7]]):
        T = len(rows)
        idx = np.asarray(rows, dtype=np.int32)
        w = np.full((T, 4), 0.5, dtype=np.float32)
        full, experts = _nvfp4_experts(shape, [0, 1, 2, 5, 7], 4)
        u = synth.activations(T, shape.hidden, 4, "u", DEV)
        out = torch.empty((T, shape.hidden), dtype=torch.bfloat16, device=DEV)
        B.beam_get_device_status()
        B.beam_moe_nvfp4(cfg, u, torch.from_numpy(idx).to(DEV), torch.from_numpy(w).to(DEV),
                         full, out, ws_for(cfg, T))
        assert B.beam_get_device_status() & B.DEV_BAD_EXPERT
        for t in range(T):
            keep = [j for j in range(4) if 0 <= rows[t][j] < shape.n_experts]
            ref = O.moe_nvfp4(shape, np64(u[t:t + 1]), idx[t:t + 1, keep],
                              np.full((1, len(keep)), 0.5), experts)
            assert_close(np64(out[t:t + 1]), ref, "moe nvfp4 out, valid slots")


def _fp8_experts(shape, used, seed):
    """FP8 expert tensors on the device (only the used experts drawn, the rest zero) and the
    oracle's view of the used ones (codes and block scales)."""
    E = shape.n_experts
    part = synth.expert_weights_fp8(shape, 0, seed, device=DEV, experts=used)
    full = {k: torch.zeros((E,) + tuple(v.shape[1:]), dtype=v.dtype, device=DEV)
            for k, v in part.items()}
    for i, e in enumerate(used):
        for k in full:
            full[k][e] = part[k][i]
    host = {k: v.cpu().numpy() for k, v in part.items()}
    experts = {e: (host["gate_up"][i], host["gate_up_scale"][i], host["down"][i],
                   host["down_scale"][i]) for i, e in enumerate(used)}
    return full, experts


@pytest.mark.parametrize("shape,T,n_used", [(TINY, 1, None), (TINY, 3, 5), (TINY, 5, None),
                                            (TINY, 13, None), (TINY, 31, 6), (BEAM, 1, None),
                                            (BEAM, 2, None), (BEAM, 4, None), (BEAM, 8, None),
                                            (BEAM, 31, 20), (TINY, 32, None), (TINY, 300, None),
                                            (NVFP4_WIDE, 130, 37), (BEAM, 48, 9)])
def test_moe_fp8(shape, T, n_used):
    """Block-scaled FP8 expert weights (e4m3 codes, one FP32 scale per 128 x 128 block):
    below 32 tokens mma.sync f16 products of the exactly converted codes, each block's sum
    times its scale; up to 4 tokens four warps split each row block's K (T=4 and T=5 sit on
    either side); T=31 over 6 experts gives experts more than 8 pairs (several passes). From
    32 tokens the grouped tensor-core GEMMs on each weight's BF16 high and low parts (130
    tokens over 37 experts: five chunks of 8; 48 full-width tokens over 9: two)."""
    seed = 97 + T
    cfg = cfg_of(shape)
    idx, w = _random_routing(shape, T, seed, n_used)
    used = sorted(set(idx.ravel().tolist()))
    full, experts = _fp8_experts(shape, used, seed)
    u = synth.activations(T, shape.hidden, seed, "u", DEV)
    out = torch.empty((T, shape.hidden), dtype=torch.bfloat16, device=DEV)
    B.beam_moe_fp8(cfg, u, torch.from_numpy(idx).to(DEV), torch.from_numpy(w).to(DEV), full,
                   out, ws_for(cfg, T))
    check_status()
    ref = O.moe_fp8(shape, np64(u), idx, w.astype(np.float64), experts)
    assert_close(np64(out), ref, "moe fp8 out")


def test_moe_fp8_bad_expert_slots_flagged_and_skipped():
    shape = TINY
    cfg = cfg_of(shape)
    for rows in ([[0, 1, 99, 2]], [[0, 1, 99, 2], [5, -3, 1, 7]]):
        T = len(rows)
        idx = np.asarray(rows, dtype=np.int32)
        w = np.full((T, 4), 0.5, dtype=np.float32)
        full, experts = _fp8_experts(shape, [0, 1, 2, 5, 7], 4)
        u = synth.activations(T, shape.hidden, 4, "u", DEV)
        out = torch.empty((T, shape.hidden), dtype=torch.bfloat16, device=DEV)
        B.beam_get_device_status()
        B.beam_moe_fp8(cfg, u, torch.from_numpy(idx).to(DEV), torch.from_numpy(w).to(DEV),
                       full, out, ws_for(cfg, T))
        assert B.beam_get_device_status() & B.DEV_BAD_EXPERT
        for t in range(T):
            keep = [j for j in range(4) if 0 <= rows[t][j] < shape.n_experts]
            ref = O.moe_fp8(shape, np64(u[t:t + 1]), idx[t:t + 1, keep],
                            np.full((1, len(keep)), 0.5), experts)
            assert_close(np64(out[t:t + 1]), ref, "moe fp8 out, valid slots")


@pytest.mark.parametrize("shape,T", [(TINY, 1), (TINY, 5), (TINY, 13), (TINY, 64), (TINY, 200),
                                     (BEAM, 1), (BEAM, 3), (BEAM, 8), (BEAM, 40), (BEAM, 130)])
def test_dense_mlp(shape, T):
    """SIMT weight streaming for one token and above 8, mma.sync row blocks for 2 to 8 tokens,
    tensor-core GEMMs from 64 tokens."""
    seed = 77 + T
    cfg = cfg_of(shape)
    Wd = synth.dense_weights(shape, 0, seed, device=DEV)
    u = synth.activations(T, shape.hidden, seed, "u", DEV)
    out = torch.empty((T, shape.hidden), dtype=torch.bfloat16, device=DEV)
    B.beam_dense_mlp(cfg, u, Wd["w_gate_up"], Wd["w_down"], out, ws_for(cfg, T))
    ref = O.dense_mlp(shape, np64(u), np64(Wd["w_gate_up"]), np64(Wd["w_down"]))
    assert_close(np64(out), ref, "dense out")


@pytest.mark.parametrize("hidden,d_ff", [(2304, 2816), (4352, 3328)])
def test_dense_mlp_one_token_ragged_rows(hidden, d_ff):
    """One token on the balanced one-CTA-per-SM kernels with widths that split rows and
    gate/up pairs unevenly over the CTAs and their warps (rows of 9-17 steps of 32 chunks; group
    counts not multiples of the SM count)."""
    shape = dataclasses.replace(BEAM, hidden=hidden, d_ff_dense=d_ff)
    cfg = cfg_of(shape)
    Wd = synth.dense_weights(shape, 0, 5, device=DEV)
    u = synth.activations(1, hidden, 5, "u", DEV)
    out = torch.empty((1, hidden), dtype=torch.bfloat16, device=DEV)
    B.beam_dense_mlp(cfg, u, Wd["w_gate_up"], Wd["w_down"], out, ws_for(cfg, 1))
    check_status()
    ref = O.dense_mlp(shape, np64(u), np64(Wd["w_gate_up"]), np64(Wd["w_down"]))
    assert_close(np64(out), ref, "dense out")


# ------------------------------------------------------------------ device-side checks ----

def test_bad_positions_are_flagged_and_skipped():
    shape = TINY
    cfg = cfg_of(shape, nope=True)
    W, u, kc, seq, pos = _qkv_inputs(shape, 2, 3, [5, 9], [0, 0], False, True)
    before = kc.k.clone()
    bad = torch.tensor([0, 10_000], dtype=torch.int32, device=DEV)   # p < 1; p > capacity
    q = torch.empty((2, shape.n_q, shape.head_dim), dtype=torch.bfloat16, device=DEV)
    g = torch.empty((2, shape.q_rows), dtype=torch.bfloat16, device=DEV)
    B.beam_get_device_status()
    B.beam_qkv_gate(cfg, u, W["w_qkvg"], W["q_norm"], W["k_norm"], seq, bad, q, g, kc,
                    ws_for(cfg, 2))
    assert B.beam_get_device_status() & B.DEV_BAD_POSITION
    assert torch.equal(kc.k, before)
    bad_seq = torch.tensor([0, 7], dtype=torch.int32, device=DEV)
    B.beam_qkv_gate(cfg, u, W["w_qkvg"], W["q_norm"], W["k_norm"], bad_seq, pos, q, g, kc,
                    ws_for(cfg, 2))
    assert B.beam_get_device_status() & B.DEV_BAD_SEQ
    # one token (its slots used directly) and two tokens (through the expert plan): the slot
    # with an out-of-range expert is flagged and left out of the combine
    wgu, wdn = synth.expert_weights(shape, 0, 1, device=DEV)
    for rows in ([[0, 1, 99, 2]], [[0, 1, 99, 2], [5, -3, 1, 7]]):
        idx = torch.tensor(rows, dtype=torch.int32, device=DEV)
        T = idx.shape[0]
        w = torch.full((T, 4), 0.5, dtype=torch.float32, device=DEV)
        out = torch.empty((T, shape.hidden), dtype=torch.bfloat16, device=DEV)
        B.beam_moe(cfg_of(shape), u[:T], idx, w, wgu, wdn, out, ws_for(cfg, T))
        assert B.beam_get_device_status() & B.DEV_BAD_EXPERT
        for t in range(T):
            keep = [j for j in range(4) if 0 <= rows[t][j] < shape.n_experts]
            ref = O.moe(shape, np64(u[t:t + 1]), np.asarray([[rows[t][j] for j in keep]]),
                        np.full((1, len(keep)), 0.5), np64(wgu), np64(wdn))
            assert_close(np64(out[t:t + 1]), ref, "moe out, valid slots")


def test_bad_positions_flagged_in_the_tensor_core_projection():
    """The prefill projection (tensor-core GEMM with the norm/RoPE/cache epilogue, 64 tokens at
    full width) flags a position < 1, a position past a NoPE cache and an out-of-range
    sequence, and writes only the valid tokens' cache slots."""
    shape, T = BEAM, 64
    cfg = cfg_of(shape, nope=True)
    positions = list(range(1, T + 1))
    W, u, kc, seq, pos = _qkv_inputs(shape, T, 4, positions, [0] * T, False, True)
    before_k, before_v = kc.k.clone(), kc.v.clone()
    bad_pos = pos.clone()
    bad_pos[3], bad_pos[10] = 0, 1_000_000
    bad_seq = seq.clone()
    bad_seq[20] = 5
    q = torch.empty((T, shape.n_q, shape.head_dim), dtype=torch.bfloat16, device=DEV)
    g = torch.empty((T, shape.q_rows), dtype=torch.bfloat16, device=DEV)
    B.beam_get_device_status()
    B.beam_qkv_gate(cfg, u, W["w_qkvg"], W["q_norm"], W["k_norm"], bad_seq, bad_pos, q, g, kc,
                    ws_for(cfg, T, T))
    bits = B.beam_get_device_status()
    assert bits & B.DEV_BAD_POSITION and bits & B.DEV_BAD_SEQ
    written = set(p - 1 for i, p in enumerate(positions) if i not in (3, 10, 20))
    untouched = [sl for sl in range(kc.k.shape[2]) if sl not in written]
    assert torch.equal(kc.k[:, :, untouched], before_k[:, :, untouched])
    assert torch.equal(kc.v[:, :, untouched], before_v[:, :, untouched])
    assert not torch.equal(kc.k[:, :, sorted(written)], before_k[:, :, sorted(written)])


def test_invalid_arguments_return_errors():
    shape = TINY
    cfg = cfg_of(shape)
    h = torch.zeros((2, 100), dtype=torch.bfloat16, device=DEV)     # H not a multiple of 8
    with pytest.raises(B.BeamError, match="invalid argument"):
        B.beam_boundary_norm(None, h, h, None, h[0], 1, 1e-6)
    x = torch.zeros((2, 256), dtype=torch.bfloat16, device=DEV)
    tiny_ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(B.BeamError, match="invalid argument"):
        Wd = synth.dense_weights(shape, 0, 1, device=DEV)
        B.beam_dense_mlp(cfg, x, Wd["w_gate_up"], Wd["w_down"], x, tiny_ws)
    bad = B.LayerCfg.from_shape(shape, B.BEAM_ATTN_SWA_ROPE)
    bad.head_dim = 96
    W = synth.attention_weights(shape, 0, 1, device=DEV)
    c = synth.kv_cache(shape, 1, 32, 1, device=DEV)
    kc = B.KVCache(c["k"], c["v"], 16)
    s = torch.zeros(2, dtype=torch.int32, device=DEV)
    with pytest.raises(B.BeamError, match="unsupported"):
        B.beam_qkv_gate(bad, x, W["w_qkvg"], W["q_norm"], W["k_norm"], s, s + 1,
                        torch.empty((2, 4, 96), dtype=torch.bfloat16, device=DEV),
                        torch.empty((2, 384), dtype=torch.bfloat16, device=DEV), kc,
                        ws_for(cfg, 2))


def test_expired_device_wait_is_reported_and_the_context_survives():
    """The bounded mbarrier wait of the tensor-core and TMA kernels, run on a barrier that
    nothing completes (no copy or MMA in flight), gives up, records DEV_TIMEOUT, and the next
    call on the device works."""
    import time
    B.beam_get_device_status()
    t0 = time.perf_counter()
    B.beam_selftest_wait_timeout()
    assert B.beam_get_device_status() & B.DEV_TIMEOUT
    print(f"bounded wait expired after {time.perf_counter() - t0:.2f} s")
    assert B.beam_get_device_status() == 0            # reading cleared it
    shape = BEAM
    x = synth.activations(2, shape.hidden, 5, "x", DEV)
    h = synth.activations(2, shape.hidden, 5, "h", DEV)
    u = torch.empty_like(h)
    w = synth.normal((shape.hidden,), 0.1, 1.0, 5, ("w",), DEV)
    h0 = np64(h)
    B.beam_boundary_norm(x, h, u, w, w, 4, shape.eps)
    check_status()
    hr, ur = O.boundary_norm(np64(x), h0, np64(w), np64(w), 4, shape.eps)
    assert_close(np64(h), hr, "h after the expired wait")
    assert_close(np64(u), ur, "u after the expired wait")
