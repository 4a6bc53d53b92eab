"""Layer and truncated-stack driver: issues the library calls of a Beam decoder layer in order.

Host orchestration only (buffer management and call order); the arithmetic is in libbeam.so.
Beam page: layers alternate sliding-window (RoPE) and NoPE full attention with every 6th layer
and the last one NoPE ("Attention" section); each sublayer sits between a post-norm and the
next pre-norm with the n-th residual term h <- sqrt((n-1)/n) h + x/sqrt(n), the embedding
being term 1 ("MoE and residual stream" section); layers 0-2 use the dense SwiGLU MLP.
"""
from __future__ import annotations

import torch

from . import beam as B


def is_nope_layer(layer: int, n_layers: int) -> bool:
    """Every 6th layer (0-based l with (l+1) % 6 == 0) and the last layer are NoPE."""
    return (layer + 1) % 6 == 0 or layer == n_layers - 1


class BeamStack:
    """A truncated Beam stack on one GPU.

    weights: list (one per layer) of dicts of device tensors, keys as made by
             synth.layer_weights (attn_pre, attn_post, mlp_pre, mlp_post, w_qkvg, q_norm,
             k_norm, gate_bias, w_o, and w_gate_up/w_down (+ router, corr_bias on MoE layers);
             an MoE layer may hold "nvfp4" (synth.expert_weights_nvfp4) or "fp8"
             (synth.expert_weights_fp8) instead of w_gate_up/w_down, and then runs
             beam_moe_nvfp4 or beam_moe_fp8).
    caches : list of B.KVCache, one per layer (window = W on sliding-window layers, 0 on NoPE).
    """

    def __init__(self, shape, weights, caches, first_layer=0, n_layers=None, device="cuda"):
        """weights[i] / caches[i] belong to global layer first_layer + i of an n_layers-deep
        stack (n_layers defaults to shape.n_layers); the layer index fixes the attention
        kind, the MLP kind and the residual term indices."""
        self.shape = shape
        self.W = weights
        self.caches = caches
        self.L = len(weights)
        self.first = first_layer
        total = shape.n_layers if n_layers is None else n_layers
        self.ids = [first_layer + i for i in range(self.L)]
        self.dense = [l in shape.dense_layers for l in self.ids]
        self.cfgs = [B.LayerCfg.from_shape(
            shape, B.BEAM_ATTN_NOPE_SSMAX if is_nope_layer(l, total) else B.BEAM_ATTN_SWA_ROPE)
            for l in self.ids]
        self.ws = B.Workspace(device)
        self.device = device
        self._bufs = {}

    def buffers(self, T):
        b = self._bufs.get(T)
        if b is None:
            s, dev = self.shape, self.device
            bf = torch.bfloat16
            b = {
                "h": torch.empty((T, s.hidden), dtype=bf, device=dev),
                "u": torch.empty((T, s.hidden), dtype=bf, device=dev),
                "q": torch.empty((T, s.n_q, s.head_dim), dtype=bf, device=dev),
                "g": torch.empty((T, s.q_rows), dtype=bf, device=dev),
                "a": torch.empty((T, s.hidden), dtype=bf, device=dev),
                "m": torch.empty((T, s.hidden), dtype=bf, device=dev),
                "logits": torch.empty((T, s.n_experts), dtype=torch.float32, device=dev),
                "idx": torch.empty((T, s.topk), dtype=torch.int32, device=dev),
                "w": torch.empty((T, s.topk), dtype=torch.float32, device=dev),
            }
            self._bufs = {T: b}
        return b

    def layer(self, i, b, seq_id, pos, max_pos, ws, stream=None, trace=None, max_q_per_seq=None):
        """The i-th layer held (global index l): from (h, u = its attention pre-norm) to
        (h, u of the next layer). With a trace list, appends the layer's intermediate tensors:
        u_attn, q, g, attn, h_mid (h after the attention residual), mlp_in, mlp, route
        (logits, idx, w) on MoE layers, and the output h."""
        W, cfg, kc = self.W[i], self.cfgs[i], self.caches[i]
        l = self.ids[i]
        if trace is not None:
            trace.append({"u_attn": b["u"].clone()})
        B.beam_qkv_gate(cfg, b["u"], W["w_qkvg"], W["q_norm"], W["k_norm"], seq_id, pos, b["q"],
                        b["g"], kc, ws, stream)
        B.beam_attn(cfg, b["q"], b["g"], W["gate_bias"], kc, seq_id, pos, max_pos, W["w_o"],
                    b["a"], ws, stream, max_q_per_seq)
        B.beam_boundary_norm(b["a"], b["h"], b["u"], W["attn_post"], W["mlp_pre"], 2 * l + 2,
                             cfg.eps, stream)
        if trace is not None:
            trace[-1].update({"q": b["q"].clone(), "g": b["g"].clone(), "attn": b["a"].clone(),
                              "h_mid": b["h"].clone(), "mlp_in": b["u"].clone()})
        if self.dense[i]:
            B.beam_dense_mlp(cfg, b["u"], W["w_gate_up"], W["w_down"], b["m"], ws, stream)
        else:
            B.beam_route(cfg, b["u"], W["router"], W["corr_bias"], b["logits"], b["idx"], b["w"],
                         ws, stream)
            if "nvfp4" in W:
                B.beam_moe_nvfp4(cfg, b["u"], b["idx"], b["w"], W["nvfp4"], b["m"], ws, stream)
            elif "fp8" in W:
                B.beam_moe_fp8(cfg, b["u"], b["idx"], b["w"], W["fp8"], b["m"], ws, stream)
            else:
                B.beam_moe(cfg, b["u"], b["idx"], b["w"], W["w_gate_up"], W["w_down"], b["m"],
                           ws, stream)
        if trace is not None:
            trace[-1]["mlp"] = b["m"].clone()
            if not self.dense[i]:
                trace[-1]["route"] = (b["logits"].clone(), b["idx"].clone(), b["w"].clone())
        nxt = self.W[i + 1]["attn_pre"] if i + 1 < self.L else None
        B.beam_boundary_norm(b["m"], b["h"], b["u"] if nxt is not None else None,
                             W["mlp_post"], nxt, 2 * l + 3, cfg.eps, stream)
        if trace is not None:
            trace[-1]["h"] = b["h"].clone()

    def forward(self, e, seq_id, pos, max_pos, stream=None, trace=None, max_q_per_seq=None):
        """Runs the held layers for the tokens (seq_id, pos). e [T][H] (bf16) is the residual
        stream entering the first held layer (the embedding when first_layer is 0); it gets
        its pre-norm first. max_q_per_seq: most tokens of one sequence (1 for a decode batch;
        None = T). Returns h after the last residual addition (an internal buffer)."""
        T = e.shape[0]
        b = self.buffers(T)
        ws = self.ws.get(B.workspace_bytes(self.cfgs[0], T, max_pos))
        b["h"].copy_(e)
        B.beam_boundary_norm(None, b["h"], b["u"], None, self.W[0]["attn_pre"], 1,
                             self.cfgs[0].eps, stream)
        for i in range(self.L):
            self.layer(i, b, seq_id, pos, max_pos, ws, stream, trace, max_q_per_seq)
        return b["h"]
