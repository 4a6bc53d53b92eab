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
from parity import (assert_chained_close, flatten_trace, noise_floor, np64, oracle_cache,
                    route_margin_ok)

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


def _check_routing(gpu_tr, ref_tr):
    for l, (g, r) in enumerate(zip(gpu_tr, ref_tr)):
        if r["route"] is not None:
            lg, idx, w = r["route"]
            gl, gi, gw = g["route"]
            assert np.array_equal(np.sort(gi.cpu().numpy(), 1), np.sort(idx, 1)), f"layer {l} idx"


def test_tiny_stack_prefill_then_decode():
    """Chained steps: each output is held to the stated bars, or to 3x the oracle's own
    divergence under FP32-level perturbation of its rounding points where that is larger;
    routing must be identical, on inputs whose routing margins exceed 10x the perturbation's
    effect on the router scores."""
    shape = TINY
    L = shape.n_layers
    caps = [128 if O.is_nope_layer(l, L) else 80 for l in range(L)]
    wins = [0 if O.is_nope_layer(l, L) else shape.window for l in range(L)]
    for seed in range(30):
        Wt = [synth.layer_weights(shape, l, seed) for l in range(L)]
        Wo = [{k: np64(v) for k, v in W.items()} for W in Wt]
        e = synth.activations(64, shape.hidden, seed, "embed")
        e1 = synth.activations(1, shape.hidden, seed, "embed_decode")
        keep = {}

        def run():
            oc = [O.KVCache(np.zeros((1, shape.n_kv, caps[l], shape.head_dim), np.float32),
                            np.zeros((1, shape.n_kv, caps[l], shape.head_dim), np.float32),
                            window=wins[l]) for l in range(L)]
            tp, td = [], []
            hp = O.stack_forward(shape, Wo, oc, np64(e), np.zeros(64, int), np.arange(1, 65), tp)
            hd = O.stack_forward(shape, Wo, oc, np64(e1), [0], [65], td)
            keep.setdefault("tr", (tp, td))
            out = flatten_trace(tp, hp, "pre.")
            out.update(flatten_trace(td, hd, "dec."))
            return out

        ref, floors = noise_floor(run)
        tr_pre, tr_dec = keep["tr"]
        fl_pre = {k[4:]: v for k, v in floors.items() if k.startswith("pre.")}
        fl_dec = {k[4:]: v for k, v in floors.items() if k.startswith("dec.")}
        if route_margin_ok(shape, tr_pre, Wo, fl_pre) and route_margin_ok(shape, tr_dec, Wo, fl_dec):
            break
    else:
        pytest.fail("no draw with routing margins above the perturbation level")
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
    _check_routing(g_pre, tr_pre)
    _check_routing(g_dec, tr_dec)
    got = flatten_trace(g_pre, h1, "pre.")
    got.update(flatten_trace(g_dec, h2, "dec."))
    assert_chained_close(got, ref, floors)


def _layer_case(shape, layer, contexts, fp8=False, scale=(1.0, 1.0)):
    """One MoE layer of the truncated stack, one decode token per sequence, chained-step bars."""
    nope = O.is_nope_layer(layer, shape.n_layers)
    S = len(contexts)
    seqs = list(range(S))
    positions = [c + 1 for c in contexts]
    max_pos = max(positions)
    cap, window = (max_pos + 8, 0) if nope else (shape.window, shape.window)
    for seed in range(10):
        W = synth.layer_weights(shape, layer, seed, device=DEV)
        c = synth.kv_cache(shape, S, cap, seed, layer, fp8=fp8, k_scale=scale[0],
                           v_scale=scale[1], device=DEV)
        kc = B.KVCache(c["k"], c["v"], window, *scale)
        oc0 = oracle_cache(kc)
        h = synth.activations(S, shape.hidden, seed, "h", DEV)
        Wo = oracle_weights(W)
        keep = {}

        def run():
            oc = O.KVCache(oc0.k, oc0.v, oc0.dtype, oc0.k_scale, oc0.v_scale, oc0.window)
            ho, uo = O.boundary_norm(None, np64(h), None, Wo["attn_pre"], 1, shape.eps)
            tr = []
            out = O.layer_forward(shape, layer, Wo, ho, uo, oc, seqs, positions, None, tr)[0]
            keep.setdefault("tr", tr)
            return flatten_trace(tr, out)

        ref, floors = noise_floor(run)
        if route_margin_ok(shape, keep["tr"], [Wo], floors):
            break
        del W, c, kc
    else:
        pytest.fail("no draw with routing margins above the perturbation level")
    st = BeamStack(shape, [W], [kc], first_layer=layer)
    gtr = []
    out = st.forward(h, torch.tensor(seqs, dtype=torch.int32, device=DEV),
                     torch.tensor(positions, dtype=torch.int32, device=DEV), max_pos, trace=gtr)
    assert B.beam_get_device_status() == 0
    _check_routing(gtr, keep["tr"])
    # the layer's output h gets the stated bar outright when the oracle is that stable
    assert_chained_close(flatten_trace(gtr, out), ref, floors, fp8)


def test_full_width_swa_moe_layer_decode_ctx4096():
    _layer_case(BEAM, 3, [4096])


@pytest.mark.parametrize("batch", [1, 8])
def test_full_width_nope_moe_layer_decode_ctx100k_bf16(batch):
    _layer_case(BEAM, 5, [100_000] * batch)


def test_full_width_nope_moe_layer_decode_ctx100k_fp8():
    _layer_case(BEAM, 5, [100_000, 100_000], fp8=True, scale=(0.0371, 0.0371))
