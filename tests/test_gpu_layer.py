"""GPU parity of single full-width layers against the oracle (the whole stack, end to end,
is in test_gpu_stack.py).

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
from synth import BEAM
from hybrid_attention_moe_gb300 import beam as B
from hybrid_attention_moe_gb300.stack import BeamStack
from parity import (assert_chained_close, assert_close, assert_logits_close, np64, oracle_cache,
                    routing_stable)

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


class LazyNvfp4:
    """expert -> its six NVFP4 arrays (oracle.moe_nvfp4), copied to the host on first use."""

    def __init__(self, d):
        self.d, self.c = d, {}

    def __getitem__(self, e):
        if e not in self.c:
            h = {k: v[e].cpu().numpy() for k, v in self.d.items()}
            self.c[e] = (h["gate_up"], h["gate_up_scale"], float(h["gate_up_global"]),
                         h["down"], h["down_scale"], float(h["down_global"]))
        return self.c[e]


class LazyFp8:
    """expert -> its four FP8 arrays (oracle.moe_fp8), copied to the host on first use."""

    def __init__(self, d):
        self.d, self.c = d, {}

    def __getitem__(self, e):
        if e not in self.c:
            h = {k: v[e].cpu().numpy() for k, v in self.d.items()}
            self.c[e] = (h["gate_up"], h["gate_up_scale"], h["down"], h["down_scale"])
        return self.c[e]


def oracle_weights(W):
    out = {}
    for k, v in W.items():
        if k == "nvfp4":
            out["nvfp4_experts"] = LazyNvfp4(v)
        elif k == "fp8":
            out["fp8_experts"] = LazyFp8(v)
        elif k in ("w_gate_up", "w_down") and v.dim() == 3:
            out[k] = LazyRows(v)
        else:
            out[k] = np64(v)
    return out


def _layer_case(shape, layer, contexts, fp8=False, scale=(1.0, 1.0), seed=0, nvfp4=False,
                fp8_experts=False):
    """One MoE layer of the truncated stack, one decode token per sequence, chained-step bars.

    The oracle runs in two stages with the oracle's own functions, in layer_forward's order:
    the attention half (to the MLP pre-norm u) once plainly and twice under FP32-level
    perturbation; then a router draw is chosen whose margins on the plain u exceed 4x the
    score shift the perturbed u causes; then the MLP half runs for all three."""
    from oracle.noise import perturbed_rounding
    from parity import max_abs_rel, mean_rel
    nope = O.is_nope_layer(layer, shape.n_layers)
    S = len(contexts)
    seqs = list(range(S))
    positions = [c + 1 for c in contexts]
    max_pos = max(positions)
    cap, window = (max_pos + 8, 0) if nope else (shape.window, shape.window)
    W = synth.layer_weights(shape, layer, seed, device=DEV,
                            with_experts=not (nvfp4 or fp8_experts))
    if nvfp4:
        W["nvfp4"] = synth.expert_weights_nvfp4(shape, layer, seed, device=DEV)
    if fp8_experts:
        W["fp8"] = synth.expert_weights_fp8(shape, layer, seed, device=DEV)
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
        if nvfp4:
            m = O.moe_nvfp4(shape, u1, idx, w, Wo["nvfp4_experts"])
        elif fp8_experts:
            m = O.moe_fp8(shape, u1, idx, w, Wo["fp8_experts"])
        else:
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
        lg = lambda u: u @ R["router"].T   # noqa: E731
        if routing_stable(shape, lg(base[2]), [lg(a[2]) for a in alts], R["corr_bias"]):
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
                     torch.tensor(positions, dtype=torch.int32, device=DEV), max_pos, trace=gtr,
                     max_q_per_seq=1)
    assert B.beam_get_device_status() == 0
    gi = np.sort(gtr[0]["route"][1].cpu().numpy(), 1)
    assert np.array_equal(gi, np.sort(ref_parts[1], 1)), "routing differs"
    got = {"L0.q": np64(gtr[0]["q"]), "L0.attn": np64(gtr[0]["attn"]),
           "L0.mlp": np64(gtr[0]["mlp"]), "h": np64(out)}
    assert_chained_close(got, ref, floors, fp8)

    # every step again on the GPU's own inputs, at the stated bars: the attention (+ gate and
    # o_proj) on the GPU's q and g over the cache holding the GPU's K/V of the new tokens, the
    # boundary norm on the GPU's attention output, the router and the experts on the GPU's u
    t = gtr[0]
    for s_, p_ in zip(seqs, positions):
        sl = oc0.slot(p_)
        if fp8:
            oc0.k[s_][:, sl] = kc.k[s_, :, sl].cpu().numpy()
            oc0.v[s_][:, sl] = kc.v[s_, :, sl].cpu().numpy()
        else:
            oc0.k[s_][:, sl] = kc.k[s_, :, sl].float().cpu().numpy()
            oc0.v[s_][:, sl] = kc.v[s_, :, sl].float().cpu().numpy()
    a_o = O.attention(shape, np64(t["q"]), np64(t["g"]), Wo["gate_bias"], oc0, seqs, positions,
                      Wo["w_o"])
    assert_close(np64(t["attn"]), a_o, "L0.attn (step)", fp8)
    hm_o, um_o = O.boundary_norm(np64(t["attn"]), ho, Wo["attn_post"], Wo["mlp_pre"],
                                 2 * layer + 2, shape.eps)
    assert_close(np64(t["h_mid"]), hm_o, "L0.h_mid (step)")
    assert_close(np64(t["mlp_in"]), um_o, "L0.mlp_in (step)")
    u_g = np64(t["mlp_in"])
    lg_g, idx_g, w_g = (x.cpu().numpy() for x in t["route"])
    lg_o, idx_o, _ = O.route(shape, u_g, R["router"], R["corr_bias"])
    assert_logits_close(lg_g.astype(np.float64), lg_o)
    assert np.array_equal(np.sort(idx_g, 1), np.sort(idx_o, 1)), "step: routing differs"
    if nvfp4:
        m_o = O.moe_nvfp4(shape, u_g, idx_g, w_g.astype(np.float64), Wo["nvfp4_experts"])
    elif fp8_experts:
        m_o = O.moe_fp8(shape, u_g, idx_g, w_g.astype(np.float64), Wo["fp8_experts"])
    else:
        m_o = O.moe(shape, u_g, idx_g, w_g.astype(np.float64), Wo["w_gate_up"], Wo["w_down"])
    assert_close(np64(t["mlp"]), m_o, "L0.mlp (step)")


def test_full_width_swa_moe_layer_decode_ctx4096():
    _layer_case(BEAM, 3, [4096])


@pytest.mark.parametrize("batch", [1, 2, 4, 8])
def test_full_width_nope_moe_layer_decode_ctx100k_bf16(batch):
    _layer_case(BEAM, 5, [100_000] * batch)


@pytest.mark.parametrize("batch", [1, 3])
def test_full_width_swa_moe_layer_decode_nvfp4_experts(batch):
    """The layer with NVFP4 expert weights (beam_moe_nvfp4 in the stack driver; the oracle's
    layer dequantises the selected experts)."""
    _layer_case(BEAM, 3, [4096] * batch, nvfp4=True)


def test_full_width_nope_moe_layer_decode_ctx100k_fp8():
    _layer_case(BEAM, 5, [100_000, 100_000], fp8=True, scale=(0.0371, 0.0371))


@pytest.mark.parametrize("batch", [1, 4])
def test_full_width_swa_moe_layer_decode_fp8_experts(batch):
    """The layer with block-scaled FP8 expert weights (beam_moe_fp8 in the stack driver; the
    oracle's layer dequantises the selected experts)."""
    _layer_case(BEAM, 3, [4096] * batch, fp8_experts=True)
