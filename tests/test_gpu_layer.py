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
    for seed in range(100):
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


def _layer_case(shape, layer, contexts, fp8=False, scale=(1.0, 1.0), seed=0):
    """One MoE layer of the truncated stack, one decode token per sequence, chained-step bars.

    The oracle runs in two stages with the oracle's own functions, in layer_forward's order:
    the attention half (to the MLP pre-norm u) once plainly and twice under FP32-level
    perturbation; then a router draw is chosen whose margins on the plain u exceed 4x the
    score shift the perturbed u causes; then the MLP half runs for all three."""
    from oracle.noise import perturbed_rounding
    from parity import ROUTE_MARGIN_FACTOR, max_abs_rel, mean_rel, route_margins
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
    oc0 = oracle_cache(kc)
    h = synth.activations(S, shape.hidden, seed, "h", DEV)
    Wo = oracle_weights(W)

    def attn_half():
        oc = O.KVCache(oc0.k, oc0.v, oc0.dtype, oc0.k_scale, oc0.v_scale, oc0.window)
        ho, uo = O.boundary_norm(None, np64(h), None, Wo["attn_pre"], 1, shape.eps)
        q, g = O.qkv_gate(shape, uo, Wo["w_qkvg"], Wo["q_norm"], Wo["k_norm"], seqs, positions,
                          oc, nope)
        a = O.attention(shape, q, g, Wo["gate_bias"], oc, seqs, positions, Wo["w_o"])
        h1, u1 = O.boundary_norm(a, ho, Wo["attn_post"], Wo["mlp_pre"], 2 * layer + 2, shape.eps)
        return {"q": q, "attn": a}, h1, u1

    def mlp_half(h1, u1, R):
        logits, idx, w = O.route(shape, u1, R["router"], R["corr_bias"])
        m = O.moe(shape, u1, idx, w, Wo["w_gate_up"], Wo["w_down"])
        h2, _ = O.boundary_norm(m, h1, Wo["mlp_post"], None, 2 * layer + 3, shape.eps)
        return logits, idx, w, m, h2

    base = attn_half()
    alts = []
    for s_ in (1, 2):
        with perturbed_rounding(seed=s_):
            alts.append(attn_half())
    # router draw whose routing the perturbation cannot flip
    for rseed in range(200):
        R = {k: np64(v) for k, v in synth.router_weights(shape, layer, 7000 + rseed).items()}
        sig = lambda u: 1.0 / (1.0 + np.exp(-(u @ R["router"].T)))   # noqa: E731
        shift = max(np.max(np.abs(sig(a[2]) - sig(base[2]))) for a in alts)
        gmin, emin = route_margins(shape, base[2], R["router"], R["corr_bias"])
        if min(gmin, emin) >= max(1e-6, ROUTE_MARGIN_FACTOR * shift):
            break
    else:
        pytest.fail("no router draw with margins above the perturbation level")
    ref_parts = mlp_half(base[1], base[2], R)
    alt_parts = []
    for s_, a in zip((1, 2), alts):
        with perturbed_rounding(seed=10 + s_):
            alt_parts.append(mlp_half(a[1], a[2], R))
    # the staged oracle is the layer: check against layer_forward once
    oc = O.KVCache(oc0.k, oc0.v, oc0.dtype, oc0.k_scale, oc0.v_scale, oc0.window)
    Wfull = dict(Wo, router=R["router"], corr_bias=R["corr_bias"])
    ho, uo = O.boundary_norm(None, np64(h), None, Wo["attn_pre"], 1, shape.eps)
    h_lf = O.layer_forward(shape, layer, Wfull, ho, uo, oc, seqs, positions, None)[0]
    assert np.array_equal(h_lf, ref_parts[4])

    ref = {"L0.q": base[0]["q"], "L0.attn": base[0]["attn"], "L0.mlp": ref_parts[3],
           "h": ref_parts[4]}
    floors = {}
    for k, r in ref.items():
        vals = []
        for a, ap in zip(alts, alt_parts):
            v = {"L0.q": a[0]["q"], "L0.attn": a[0]["attn"], "L0.mlp": ap[3], "h": ap[4]}[k]
            vals.append((max_abs_rel(v, r), mean_rel(v, r), float(np.max(np.abs(v - r)))))
        floors[k] = tuple(max(x[i] for x in vals) for i in range(3))

    W["router"] = torch.from_numpy(R["router"]).float().to(DEV)
    W["corr_bias"] = torch.from_numpy(R["corr_bias"]).float().to(DEV)
    st = BeamStack(shape, [W], [kc], first_layer=layer)
    gtr = []
    out = st.forward(h, torch.tensor(seqs, dtype=torch.int32, device=DEV),
                     torch.tensor(positions, dtype=torch.int32, device=DEV), max_pos, trace=gtr)
    assert B.beam_get_device_status() == 0
    gi = np.sort(gtr[0]["route"][1].cpu().numpy(), 1)
    assert np.array_equal(gi, np.sort(ref_parts[1], 1)), "routing differs"
    got = {"L0.q": np64(gtr[0]["q"]), "L0.attn": np64(gtr[0]["attn"]),
           "L0.mlp": np64(gtr[0]["mlp"]), "h": np64(out)}
    assert_chained_close(got, ref, floors, fp8)


def test_full_width_swa_moe_layer_decode_ctx4096():
    _layer_case(BEAM, 3, [4096])


@pytest.mark.parametrize("batch", [1, 8])
def test_full_width_nope_moe_layer_decode_ctx100k_bf16(batch):
    _layer_case(BEAM, 5, [100_000] * batch)


def test_full_width_nope_moe_layer_decode_ctx100k_fp8():
    _layer_case(BEAM, 5, [100_000, 100_000], fp8=True, scale=(0.0371, 0.0371))
