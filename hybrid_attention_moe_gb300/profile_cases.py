"""Small, self-contained invocations of single library calls, for profiler captures.

Each case holds at most a few GB on the device while its inputs still exceed the 129 MB L2,
and repeats the call `--reps` times after `--warmup` untimed calls, so a profiler can skip the
warm-up launches and capture one or a few real ones. Usage:

    python -m hybrid_attention_moe_gb300.profile_cases --case moe_decode --reps 3

Cases: moe_decode (--tokens tokens, default 1, each over 8 selected experts of a 32-expert
pool), moe_decode_nvfp4 / moe_decode_fp8 (the same with NVFP4 / block-scaled FP8 expert weights), dense_decode (the 20480-wide dense SwiGLU MLP for --tokens tokens),
lm_head_decode (the LM head with the logit softcap over 32768 vocabulary rows, --tokens tokens),
qkv_decode, oproj_decode (via beam_attn on a 512-key window), attn_nope_decode (100K keys),
route_decode, norm_decode, gemm_prefill (2048 x 14336 x 5120 tensor-core GEMM),
moe_prefill (grouped tensor-core GEMMs, 2048 tokens over 32 experts), attn_nope_prefill
(tensor-core attention: one sequence, 2048 new tokens after --ctx cached keys, NoPE, BF16 KV),
attn_swa_prefill (the same over a 512-key sliding window, 8 sequences), attn_nope_verify
(--tokens new tokens of one sequence after --ctx cached keys, NoPE, BF16 KV, bound = tokens:
the grouped decode form of a verification batch).
"""
from __future__ import annotations

import argparse
import dataclasses
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402
from hybrid_attention_moe_gb300 import beam as B  # noqa: E402
from hybrid_attention_moe_gb300 import build as _build  # noqa: E402


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", required=True)
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=2)
    ap.add_argument("--ctx", type=int, default=16384)
    ap.add_argument("--tokens", type=int, default=1)
    args = ap.parse_args()
    _build.build()
    dev = "cuda"
    shape = synth.BEAM
    small = dataclasses.replace(shape, n_experts=32, n_groups=8, topk_groups=4)
    cfg = B.LayerCfg.from_shape(shape, B.BEAM_ATTN_SWA_ROPE)
    H = shape.hidden
    c = args.case
    if c == "moe_decode" or c == "moe_prefill":
        T = args.tokens if c == "moe_decode" else 2048
        cs = B.LayerCfg.from_shape(small, B.BEAM_ATTN_SWA_ROPE)
        wgu, wdn = synth.expert_weights(small, 3, 0, device=dev)
        u = synth.activations(T, H, 0, "u", dev)
        g = torch.Generator(device="cpu").manual_seed(0)
        idx = torch.stack([torch.randperm(32, generator=g)[:8] for _ in range(T)]).int().to(dev)
        w = torch.full((T, 8), 0.3, device=dev)
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(B.workspace_bytes(cs, T, 1), dtype=torch.uint8, device=dev)
        fn = lambda: B.beam_moe(cs, u, idx, w, wgu, wdn, out, ws)  # noqa: E731
    elif c == "moe_decode_nvfp4":
        T = args.tokens
        cs = B.LayerCfg.from_shape(small, B.BEAM_ATTN_SWA_ROPE)
        wq = synth.expert_weights_nvfp4(small, 3, 0, device=dev)
        u = synth.activations(T, H, 0, "u", dev)
        g = torch.Generator(device="cpu").manual_seed(0)
        idx = torch.stack([torch.randperm(32, generator=g)[:8] for _ in range(T)]).int().to(dev)
        w = torch.full((T, 8), 0.3, device=dev)
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(B.workspace_bytes(cs, T, 1), dtype=torch.uint8, device=dev)
        fn = lambda: B.beam_moe_nvfp4(cs, u, idx, w, wq, out, ws)  # noqa: E731
    elif c == "moe_decode_fp8":
        T = args.tokens
        cs = B.LayerCfg.from_shape(small, B.BEAM_ATTN_SWA_ROPE)
        wq = synth.expert_weights_fp8(small, 3, 0, device=dev)
        u = synth.activations(T, H, 0, "u", dev)
        g = torch.Generator(device="cpu").manual_seed(0)
        idx = torch.stack([torch.randperm(32, generator=g)[:8] for _ in range(T)]).int().to(dev)
        w = torch.full((T, 8), 0.3, device=dev)
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(B.workspace_bytes(cs, T, 1), dtype=torch.uint8, device=dev)
        fn = lambda: B.beam_moe_fp8(cs, u, idx, w, wq, out, ws)  # noqa: E731
    elif c == "lm_head_decode":
        # 32768 vocabulary rows at hidden 5120: 336 MB of BF16 weights (more than L2)
        T, V = args.tokens, 32768
        Wh = synth.lm_head_weights(shape, V, 0, device=dev)
        u = synth.activations(T, H, 0, "u_final", dev)
        logits = torch.empty((T, V), dtype=torch.float32, device=dev)
        fn = lambda: B.beam_lm_head(u, Wh["w_lm"], logits, softcap=30.0)  # noqa: E731
    elif c == "dense_decode":
        T = args.tokens
        Wd = synth.dense_weights(shape, 0, 0, device=dev)
        u = synth.activations(T, H, 0, "u", dev)
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(B.workspace_bytes(cfg, T, 1), dtype=torch.uint8, device=dev)
        fn = lambda: B.beam_dense_mlp(cfg, u, Wd["w_gate_up"], Wd["w_down"], out, ws)  # noqa: E731
    elif c == "qkv_decode":
        W = synth.attention_weights(shape, 3, 0, device=dev)
        u = synth.activations(1, H, 0, "u", dev)
        kv = synth.kv_cache(shape, 1, shape.window, 0, device=dev)
        kc = B.KVCache(kv["k"], kv["v"], shape.window)
        q = torch.empty((1, shape.n_q, shape.head_dim), dtype=torch.bfloat16, device=dev)
        gg = torch.empty((1, shape.q_rows), dtype=torch.bfloat16, device=dev)
        seq = torch.zeros(1, dtype=torch.int32, device=dev)
        pos = torch.full((1,), 4097, dtype=torch.int32, device=dev)
        ws = torch.empty(B.workspace_bytes(cfg, 1, 4097), dtype=torch.uint8, device=dev)
        fn = lambda: B.beam_qkv_gate(cfg, u, W["w_qkvg"], W["q_norm"], W["k_norm"], seq, pos, q,  # noqa: E731
                                     gg, kc, ws)
    elif c in ("oproj_decode", "attn_nope_decode"):
        nope = c == "attn_nope_decode"
        ctx = 100_000 if nope else 4096
        cf = B.LayerCfg.from_shape(shape, B.BEAM_ATTN_NOPE_SSMAX if nope else B.BEAM_ATTN_SWA_ROPE)
        W = synth.attention_weights(shape, 5, 0, device=dev)
        cap, win = (ctx + 8, 0) if nope else (shape.window, shape.window)
        kv = synth.kv_cache(shape, 1, cap, 0, device=dev)
        kc = B.KVCache(kv["k"], kv["v"], win)
        q = synth.normal((1, shape.n_q, shape.head_dim), 1.0, 0.0, 0, ("q",), dev)
        gg = synth.activations(1, shape.q_rows, 0, "g", dev)
        seq = torch.zeros(1, dtype=torch.int32, device=dev)
        pos = torch.full((1,), ctx + 1, dtype=torch.int32, device=dev)
        out = torch.empty((1, H), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(B.workspace_bytes(cf, 1, ctx + 1), dtype=torch.uint8, device=dev)
        fn = lambda: B.beam_attn(cf, q, gg, W["gate_bias"], kc, seq, pos, ctx + 1, W["w_o"], out, ws,  # noqa: E731
                                 max_q_per_seq=1)
    elif c in ("attn_nope_prefill", "attn_swa_prefill"):
        nope = c == "attn_nope_prefill"
        S, chunk = (1, 2048) if nope else (8, 2048)
        ctx = args.ctx
        cf = B.LayerCfg.from_shape(shape, B.BEAM_ATTN_NOPE_SSMAX if nope else B.BEAM_ATTN_SWA_ROPE)
        W = synth.attention_weights(shape, 5, 0, device=dev)
        cap, win = (ctx + chunk + 8, 0) if nope else (-(-(shape.window + chunk - 1) // 128) * 128,
                                                      shape.window)
        kv = synth.kv_cache(shape, S, cap, 0, device=dev)
        kc = B.KVCache(kv["k"], kv["v"], win)
        T = S * chunk
        q = synth.normal((T, shape.n_q, shape.head_dim), 1.0, 0.0, 0, ("q",), dev)
        gg = synth.activations(T, shape.q_rows, 0, "g", dev)
        seq, pos = synth.prefill_positions([ctx] * S, chunk, dev)
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(B.workspace_bytes(cf, T, ctx + chunk), dtype=torch.uint8, device=dev)
        fn = lambda: B.beam_attn(cf, q, gg, W["gate_bias"], kc, seq, pos, ctx + chunk, W["w_o"],  # noqa: E731
                                 out, ws, max_q_per_seq=chunk)
    elif c == "attn_nope_verify":
        ctx, T = args.ctx, args.tokens
        cf = B.LayerCfg.from_shape(shape, B.BEAM_ATTN_NOPE_SSMAX)
        W = synth.attention_weights(shape, 5, 0, device=dev)
        kv = synth.kv_cache(shape, 1, ctx + T + 8, 0, device=dev)
        kc = B.KVCache(kv["k"], kv["v"], 0)
        q = synth.normal((T, shape.n_q, shape.head_dim), 1.0, 0.0, 0, ("q",), dev)
        gg = synth.activations(T, shape.q_rows, 0, "g", dev)
        seq, pos = synth.prefill_positions([ctx], T, dev)
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(B.workspace_bytes(cf, T, ctx + T), dtype=torch.uint8, device=dev)
        fn = lambda: B.beam_attn(cf, q, gg, W["gate_bias"], kc, seq, pos, ctx + T, W["w_o"], out,  # noqa: E731
                                 ws, max_q_per_seq=T)
    elif c == "route_decode":
        R = synth.router_weights(shape, 3, 0, device=dev)
        u = synth.activations(1, H, 0, "u", dev)
        lg = torch.empty((1, 256), dtype=torch.float32, device=dev)
        idx = torch.empty((1, 8), dtype=torch.int32, device=dev)
        w = torch.empty((1, 8), dtype=torch.float32, device=dev)
        ws = torch.empty(B.workspace_bytes(cfg, 1, 1), dtype=torch.uint8, device=dev)
        fn = lambda: B.beam_route(cfg, u, R["router"], R["corr_bias"], lg, idx, w, ws)  # noqa: E731
    elif c == "norm_decode":
        x = synth.activations(1, H, 0, "x", dev)
        h = synth.activations(1, H, 0, "h", dev)
        uu = torch.empty_like(h)
        wv = synth.normal((H,), 0.1, 1.0, 0, ("w",), dev)
        fn = lambda: B.beam_boundary_norm(x, h, uu, wv, wv, 8, 1e-6)  # noqa: E731
    elif c == "gemm_prefill":
        a = synth.activations(2048, H, 0, "a", dev)
        wq = synth.normal((shape.qkvg_rows, H), 0.02, 0.0, 0, ("w",), dev)
        cc = torch.empty((2048, shape.qkvg_rows), dtype=torch.float32, device=dev)
        fn = lambda: B.beam_gemm_bf16(a, wq, cc)  # noqa: E731
    else:
        raise SystemExit(f"unknown case {c}")
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    for _ in range(args.reps):
        fn()
    torch.cuda.synchronize()
    assert B.beam_get_device_status() == 0
    print(f"{c}: ok")


if __name__ == "__main__":
    main()
