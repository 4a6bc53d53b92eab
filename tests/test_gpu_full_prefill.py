"""GPU parity of every layer step at the full prefill size bench.py times: 8 sequences x 2048
new tokens (T = 16384) at full Beam width, in the same launch configuration (tensor-core
GEMMs, the tensor-core attention over 100,000 cached keys, the tensor-core router).

The oracle cannot run 16384 tokens, so each step is checked on sampled tokens (first, middle
and last of the chunk, in the first and the last sequence), which the oracle computes one by
one from the same seeded inputs. Expert weights reach the oracle only for the experts the
sampled tokens use.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from synth import BEAM
from hybrid_attention_moe_gb300 import beam as B
from parity import assert_close, assert_logits_close, np64, route_margins

pytestmark = pytest.mark.gpu
DEV = "cuda"
S, CHUNK, CTX = 8, 2048, 100_000
T = S * CHUNK
SAMPLE = [s * CHUNK + i for s in (0, S - 1) for i in (0, CHUNK // 2, CHUNK - 1)]


def cfg_of(nope):
    return B.LayerCfg.from_shape(BEAM, B.BEAM_ATTN_NOPE_SSMAX if nope else B.BEAM_ATTN_SWA_ROPE)


def ws_for(cfg, max_pos=1):
    return torch.empty(B.workspace_bytes(cfg, T, max_pos), dtype=torch.uint8, device=DEV)


def check_status():
    bits = B.beam_get_device_status()
    assert bits == 0, f"device status bits {bits:#x}"


def seq_pos():
    seq, pos = synth.prefill_positions([CTX] * S, CHUNK, DEV)
    return seq, pos, seq.cpu().numpy(), pos.cpu().numpy()


def one_seq_cache(kc, s):
    """Oracle copy of sequence s of a BF16 binding cache (index 0 of the copy)."""
    return O.KVCache(kc.k[s:s + 1].float().cpu().numpy(), kc.v[s:s + 1].float().cpu().numpy(),
                     "bf16", window=kc.window)


@pytest.mark.parametrize("nope", [True, False])
def test_full_prefill_attention_sampled(nope):
    """beam_attn over 8 x 2048 tokens: NoPE over 100,000 + chunk keys (the bench's NoPE
    layer), or the 512-key window on a 2560-slot ring."""
    cfg = cfg_of(nope)
    seq, pos, seqs, positions = seq_pos()
    max_pos = CTX + CHUNK
    cap, window = (max_pos + 8, 0) if nope else (2560, BEAM.window)
    c = synth.kv_cache(BEAM, S, cap, 5, device=DEV)
    kc = B.KVCache(c["k"], c["v"], window)
    q = synth.normal((T, BEAM.n_q, BEAM.head_dim), 1.0, 0.0, 5, ("q",), DEV)
    g = synth.activations(T, BEAM.q_rows, 5, "g", DEV)
    W = synth.attention_weights(BEAM, 5, 5, device=DEV)
    out = torch.empty((T, BEAM.hidden), dtype=torch.bfloat16, device=DEV)
    B.beam_attn(cfg, q, g, W["gate_bias"], kc, seq, pos, max_pos, W["w_o"], out,
                ws_for(cfg, max_pos), max_q_per_seq=CHUNK)
    check_status()
    wo, gb = np64(W["w_o"]), np64(W["gate_bias"])
    for s in (0, S - 1):
        oc = one_seq_cache(kc, s)
        rows = [t for t in SAMPLE if seqs[t] == s]
        ref = O.attention(BEAM, np64(q[rows]), np64(g[rows]), gb, oc, [0] * len(rows),
                          [int(positions[t]) for t in rows], wo)
        assert_close(np64(out[rows]), ref, f"attn out, sequence {s}")


@pytest.mark.parametrize("nope", [True, False])
def test_full_prefill_qkv_gate_sampled(nope):
    """beam_qkv_gate over 8 x 2048 tokens (tensor-core projection + epilogue): q', g and the
    K/V written into the cache, on the sampled tokens."""
    cfg = cfg_of(nope)
    seq, pos, seqs, positions = seq_pos()
    cap, window = (CTX + CHUNK + 8, 0) if nope else (2560, BEAM.window)
    kc = B.KVCache(torch.zeros((S, BEAM.n_kv, cap, BEAM.head_dim), dtype=torch.bfloat16, device=DEV),
                   torch.zeros((S, BEAM.n_kv, cap, BEAM.head_dim), dtype=torch.bfloat16, device=DEV),
                   window)
    W = synth.attention_weights(BEAM, 2, 7, device=DEV)
    u = synth.activations(T, BEAM.hidden, 7, "u", DEV)
    q = torch.empty((T, BEAM.n_q, BEAM.head_dim), dtype=torch.bfloat16, device=DEV)
    g = torch.empty((T, BEAM.q_rows), dtype=torch.bfloat16, device=DEV)
    B.beam_qkv_gate(cfg, u, W["w_qkvg"], W["q_norm"], W["k_norm"], seq, pos, q, g, kc,
                    ws_for(cfg, CTX + CHUNK))
    check_status()
    # the oracle's cache only needs the sampled tokens' slots: one small ring per sampled
    # token (tokens of different sequences share positions)
    ocap, n = 4096, len(SAMPLE)
    oc = O.KVCache(np.zeros((n, BEAM.n_kv, ocap, BEAM.head_dim)),
                   np.zeros((n, BEAM.n_kv, ocap, BEAM.head_dim)), "bf16", window=window)
    ps = [int(positions[t]) for t in SAMPLE]
    q_ref, g_ref = O.qkv_gate(BEAM, np64(u[SAMPLE]), np64(W["w_qkvg"]), np64(W["q_norm"]),
                              np64(W["k_norm"]), list(range(n)), ps, oc, nope)
    assert_close(np64(q[SAMPLE]), q_ref, "q'")
    assert_close(np64(g[SAMPLE]), g_ref, "g")
    for i, (t, p) in enumerate(zip(SAMPLE, ps)):
        sl, osl = (p - 1) % cap, (p - 1) % ocap
        s = int(seqs[t])
        assert_close(np64(kc.k[s, :, sl]), oc.k[i][:, osl], f"cached k, token {t}")
        assert_close(np64(kc.v[s, :, sl]), oc.v[i][:, osl], f"cached v, token {t}")


def test_full_prefill_route_sampled():
    """beam_route over 16384 tokens (logits from the exact three-part BF16 split on the
    tensor cores): logits of the sampled tokens to 1e-5, and their selection where the
    oracle's margins exceed 1e-6."""
    cfg = cfg_of(False)
    u = synth.activations(T, BEAM.hidden, 11, "u", DEV)
    R = synth.router_weights(BEAM, 3, 11, device=DEV)
    logits = torch.empty((T, BEAM.n_experts), dtype=torch.float32, device=DEV)
    idx = torch.empty((T, BEAM.topk), dtype=torch.int32, device=DEV)
    w = torch.empty((T, BEAM.topk), dtype=torch.float32, device=DEV)
    B.beam_route(cfg, u, R["router"], R["corr_bias"], logits, idx, w, ws_for(cfg))
    check_status()
    us, wr, cb = np64(u[SAMPLE]), np64(R["router"]), np64(R["corr_bias"])
    lg_ref, idx_ref, w_ref = O.route(BEAM, us, wr, cb)
    assert_logits_close(logits[SAMPLE].cpu().double().numpy(), lg_ref)
    checked = 0
    for i, t in enumerate(SAMPLE):
        gmin, emin = route_margins(BEAM, us[i:i + 1], wr, cb)
        if min(gmin, emin) < 1e-6:
            continue
        checked += 1
        assert idx[t].cpu().tolist() == idx_ref[i].tolist(), f"token {t}"
        rel = np.abs(w[t].cpu().double().numpy() - w_ref[i]) / np.abs(w_ref[i])
        assert rel.max() < 1e-5
    assert checked >= len(SAMPLE) // 2


def test_full_prefill_moe_sampled():
    """beam_moe over 16384 tokens x 8 slots on all 256 experts (grouped tensor-core GEMMs),
    seeded uniform routing; the sampled tokens' combined rows."""
    cfg = cfg_of(False)
    rng = np.random.default_rng(13)
    idx = np.stack([rng.choice(BEAM.n_experts, BEAM.topk, replace=False) for _ in range(T)])
    wts = rng.uniform(0.05, 0.6, size=(T, BEAM.topk)).astype(np.float32)
    wgu, wdn = synth.expert_weights(BEAM, 3, 13, device=DEV)
    u = synth.activations(T, BEAM.hidden, 13, "u", DEV)
    out = torch.empty((T, BEAM.hidden), dtype=torch.bfloat16, device=DEV)
    B.beam_moe(cfg, u, torch.from_numpy(idx.astype(np.int32)).to(DEV),
               torch.from_numpy(wts).to(DEV), wgu, wdn, out, ws_for(cfg))
    check_status()
    # one token at a time: only its 8 experts are copied to the host
    for t in (SAMPLE[0], SAMPLE[2], SAMPLE[3], SAMPLE[5]):
        ogu = {int(e): np64(wgu[int(e)]) for e in idx[t]}
        odn = {int(e): np64(wdn[int(e)]) for e in idx[t]}
        ref = O.moe(BEAM, np64(u[t:t + 1]), idx[t:t + 1], wts[t:t + 1].astype(np.float64),
                    ogu, odn)
        assert_close(np64(out[t:t + 1]), ref, f"moe out, token {t}")


def test_full_prefill_dense_mlp_sampled():
    """beam_dense_mlp over 16384 tokens (SwiGLU-epilogue GEMM, then the down GEMM)."""
    cfg = cfg_of(False)
    Wd = synth.dense_weights(BEAM, 0, 17, device=DEV)
    u = synth.activations(T, BEAM.hidden, 17, "u", DEV)
    out = torch.empty((T, BEAM.hidden), dtype=torch.bfloat16, device=DEV)
    B.beam_dense_mlp(cfg, u, Wd["w_gate_up"], Wd["w_down"], out, ws_for(cfg))
    check_status()
    ref = O.dense_mlp(BEAM, np64(u[SAMPLE]), np64(Wd["w_gate_up"]), np64(Wd["w_down"]))
    assert_close(np64(out[SAMPLE]), ref, "dense out")
