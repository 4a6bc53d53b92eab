"""GPU parity of whole layers and of the truncated stack against the oracle.

  - tiny 6-layer stack (hidden 256, 4/2 heads of 64, window 16, 16 experts; layer 0 dense,
    layer 5 NoPE): prefill of 64 N(0,1) tokens through every layer (filling every cache),
    then one decode token at p = 65;
  - one full-width sliding-window MoE layer, batch-1 decode at context 4096 (BF16 cache);
  - one full-width NoPE MoE layer with SSMax, decode at context 100,000 per sequence,
    batch 1 and 8 with a BF16 cache, batch 2 with an FP8-e4m3 cache (scale 0.0371).
Every input is drawn by `synth`; expert weights reach the oracle only for the experts its
own routing selects.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from synth import BEAM, TINY
from hybrid_attention_moe_gb300 import beam as B
from hybrid_attention_moe_gb300.stack import BeamStack
from parity import assert_close, assert_logits_close, np64, oracle_cache, route_margins

pytestmark = pytest.mark.gpu
DEV = "cuda"


class LazyRows:
    """expert index -> float64 host copy of that expert's weights, fetched on first use."""

    def __init__(self, t):
        self.t = t
        self.cache = {}

    def __getitem__(self, e):
        if e not in self.cache:
            self.cache[e] = np64(self.t[e])
        return self.cache[e]


def oracle_weights(W):
    out = {}
    for k, v in W.items():
        if k in ("w_gate_up", "w_down") and v.dim() == 3:
            out[k] = LazyRows(v)
        else:
            out[k] = np64(v)
    return out


def _check_trace(gpu_tr, ref_tr, fp8=False):
    for l, (g, r) in enumerate(zip(gpu_tr, ref_tr)):
        assert_close(np64(g["q"]), r["q"], f"layer {l} q'", fp8)
        assert_close(np64(g["attn"]), r["attn"], f"layer {l} attention out", fp8)
        assert_close(np64(g["mlp"]), r["mlp"], f"layer {l} mlp out", fp8)
        if r["route"] is not None:
            lg, idx, w = r["route"]
            gl, gi, gw = g["route"]
            assert_logits_close(gl.cpu().double().numpy(), lg, f"layer {l} logits")
            assert np.array_equal(np.sort(gi.cpu().numpy(), 1), np.sort(idx, 1)), f"layer {l} idx"


def _min_margin(shape, W, trace):
    m = np.inf
    for l, tr in enumerate(trace):
        if tr["route"] is not None:
            g, e = route_margins(shape, tr["mlp_in"], W[l]["router"], W[l]["corr_bias"])
            m = min(m, g, e)
    return m


def test_tiny_stack_prefill_then_decode():
    shape = TINY
    L = shape.n_layers
    for seed in range(20):
        Wt = [synth.layer_weights(shape, l, seed) for l in range(L)]
        Wo = [{k: np64(v) for k, v in W.items()} for W in Wt]
        e = synth.activations(64, shape.hidden, seed, "embed")
        e1 = synth.activations(1, shape.hidden, seed, "embed_decode")
        caps = [128 if O.is_nope_layer(l, L) else 80 for l in range(L)]
        wins = [0 if O.is_nope_layer(l, L) else shape.window for l in range(L)]
        oc = [O.KVCache(np.zeros((1, shape.n_kv, caps[l], shape.head_dim), np.float32),
                        np.zeros((1, shape.n_kv, caps[l], shape.head_dim), np.float32),
                        window=wins[l]) for l in range(L)]
        tr_pre, tr_dec = [], []
        h_pre = O.stack_forward(shape, Wo, oc, np64(e), np.zeros(64, int), np.arange(1, 65), tr_pre)
        h_dec = O.stack_forward(shape, Wo, oc, np64(e1), [0], [65], tr_dec)
        if min(_min_margin(shape, Wo, tr_pre), _min_margin(shape, Wo, tr_dec)) >= 1e-6:
            break
    Wd = [{k: v.to(DEV) for k, v in W.items()} for W in Wt]
    caches = [B.KVCache(torch.zeros((1, shape.n_kv, caps[l], shape.head_dim), dtype=torch.bfloat16,
                                    device=DEV),
                        torch.zeros((1, shape.n_kv, caps[l], shape.head_dim), dtype=torch.bfloat16,
                                    device=DEV), wins[l]) for l in range(L)]
    st = BeamStack(shape, Wd, caches)
    g_pre, g_dec = [], []
    seq = torch.zeros(64, dtype=torch.int32, device=DEV)
    pos = torch.arange(1, 65, dtype=torch.int32, device=DEV)
    h1 = st.forward(e.to(DEV), seq, pos, 64, trace=g_pre).clone()
    h2 = st.forward(e1.to(DEV), seq[:1], torch.tensor([65], dtype=torch.int32, device=DEV), 65,
                    trace=g_dec).clone()
    assert B.beam_get_device_status() == 0
    _check_trace(g_pre, tr_pre)
    _check_trace(g_dec, tr_dec)
    assert_close(np64(h1), h_pre, "stack prefill h")
    assert_close(np64(h2), h_dec, "stack decode h")


def _one_layer(shape, layer, contexts, fp8=False, scale=(1.0, 1.0), seed=0):
    """One MoE layer `layer` of the truncated stack, one decode token per sequence."""
    nope = O.is_nope_layer(layer, shape.n_layers)
    S = len(contexts)
    seqs = list(range(S))
    positions = [c + 1 for c in contexts]
    max_pos = max(positions)
    cap, window = (max_pos + 8, 0) if nope else (shape.window, shape.window)
    W = synth.layer_weights(shape, layer, seed, device=DEV)
    c = synth.kv_cache(shape, S, cap, seed, layer, fp8=fp8, k_scale=scale[0], v_scale=scale[1],
                       device=DEV)
    kc = B.KVCache(c["k"], c["v"], window, *scale)
    oc = oracle_cache(kc)
    h = synth.activations(S, shape.hidden, seed, "h", DEV)
    Wo = oracle_weights(W)
    ho, uo = O.boundary_norm(None, np64(h), None, Wo["attn_pre"], 1, shape.eps)
    tr = []
    ref = O.layer_forward(shape, layer, Wo, ho, uo, oc, seqs, positions, None, tr)[0]
    st = BeamStack(shape, [W], [kc], first_layer=layer)
    gtr = []
    out = st.forward(h, torch.tensor(seqs, dtype=torch.int32, device=DEV),
                     torch.tensor(positions, dtype=torch.int32, device=DEV), max_pos, trace=gtr)
    assert B.beam_get_device_status() == 0
    margin = _min_margin(shape, [Wo], tr)
    return np64(out), ref, gtr, tr, margin


def _layer_case(shape, layer, contexts, fp8=False, scale=(1.0, 1.0)):
    for seed in range(10):
        out, ref, gtr, tr, margin = _one_layer(shape, layer, contexts, fp8, scale, seed)
        if margin >= 1e-6:
            break
    _check_trace(gtr, tr, fp8)
    assert_close(out, ref, "layer out h", fp8)


def test_full_width_swa_moe_layer_decode_ctx4096():
    _layer_case(BEAM, 3, [4096])


@pytest.mark.parametrize("batch", [1, 8])
def test_full_width_nope_moe_layer_decode_ctx100k_bf16(batch):
    _layer_case(BEAM, 5, [100_000] * batch)


def test_full_width_nope_moe_layer_decode_ctx100k_fp8():
    _layer_case(BEAM, 5, [100_000, 100_000], fp8=True, scale=(0.0371, 0.0371))
