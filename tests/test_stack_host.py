"""Host logic of the stack driver (stack.py) on the CPU: the binding's calls are replaced by
recorders, so no kernel runs. It checks what the driver alone decides: the order of the calls,
the residual index n of every boundary (the embedding 1, then 2, 3, ... 2L + 1, as the oracle
counts them), the last boundary without a next pre-norm, the attention kind of each layer
(NoPE every 6th and last), and which MLP call each layer makes (dense layers, routed experts,
NVFP4 experts)."""
import torch

import synth
from synth import TINY
from hybrid_attention_moe_gb300 import beam as B
from hybrid_attention_moe_gb300 import stack as S

CALLS = ["beam_qkv_gate", "beam_attn", "beam_boundary_norm", "beam_dense_mlp", "beam_route",
         "beam_moe", "beam_moe_nvfp4"]


def run_stack(monkeypatch, weights, first_layer=0, n_layers=None, T=3):
    seen = []
    for name in CALLS:
        monkeypatch.setattr(B, name, lambda *a, _n=name, **k: seen.append((_n, a)))
    monkeypatch.setattr(B, "workspace_bytes", lambda *a: 0)
    shape = TINY
    caches = [B.KVCache(torch.zeros(1), torch.zeros(1), 0) for _ in weights]
    st = S.BeamStack(shape, weights, caches, first_layer=first_layer, n_layers=n_layers,
                     device="cpu")
    e = torch.zeros((T, shape.hidden), dtype=torch.bfloat16)
    st.forward(e, torch.zeros(T, dtype=torch.int32), torch.arange(1, T + 1, dtype=torch.int32), T)
    return st, seen


def test_full_stack_call_order_and_residual_indices(monkeypatch):
    L = TINY.n_layers
    W = [synth.layer_weights(TINY, l, 0) for l in range(L)]
    st, seen = run_stack(monkeypatch, W)
    norms = [a for n, a in seen if n == "beam_boundary_norm"]
    assert [a[5] for a in norms] == list(range(1, 2 * L + 2))
    assert norms[0][0] is None                       # the embedding: pre-norm only
    assert norms[-1][2] is None and norms[-1][4] is None   # no pre-norm after the last MLP
    per_layer = []
    for n, a in seen:
        if n == "beam_qkv_gate":
            per_layer.append([])
        if per_layer:
            per_layer[-1].append(n)
    assert len(per_layer) == L
    for l, names in enumerate(per_layer):
        mlp = (["beam_dense_mlp"] if l in TINY.dense_layers else ["beam_route", "beam_moe"])
        assert names == ["beam_qkv_gate", "beam_attn", "beam_boundary_norm", *mlp,
                         "beam_boundary_norm"], (l, names)
    kinds = [a[0].kind for n, a in seen if n == "beam_attn"]
    nope = [(l + 1) % 6 == 0 or l == L - 1 for l in range(L)]
    assert kinds == [B.BEAM_ATTN_NOPE_SSMAX if x else B.BEAM_ATTN_SWA_ROPE for x in nope]


def test_held_layer_takes_global_indices_and_nvfp4_experts(monkeypatch):
    """One held MoE layer (global layer 3 of 6) with NVFP4 experts: its residual terms are
    2*3+2 = 8 and 9, it runs beam_moe_nvfp4, and its attention is sliding-window."""
    W = synth.layer_weights(TINY, 3, 0, with_experts=False)
    W["nvfp4"] = {"marker": torch.zeros(1)}
    st, seen = run_stack(monkeypatch, [W], first_layer=3, n_layers=6)
    names = [n for n, _ in seen]
    assert names == ["beam_boundary_norm", "beam_qkv_gate", "beam_attn", "beam_boundary_norm",
                     "beam_route", "beam_moe_nvfp4", "beam_boundary_norm"]
    assert [a[5] for n, a in seen if n == "beam_boundary_norm"] == [1, 8, 9]
    moe_args = [a for n, a in seen if n == "beam_moe_nvfp4"][0]
    assert moe_args[4] is W["nvfp4"]
    assert [a[0].kind for n, a in seen if n == "beam_attn"] == [B.BEAM_ATTN_SWA_ROPE]
