"""The allocation-free router variant, through the C ABI, against the regular beam_route.

beam_route_noalloc is for callers that cannot give the library device scratch (an engine that
handed all free memory to its KV-cache pool, a runtime that may not allocate once running): it
keeps the router logits in a static device array of the library instead. Two calls in a row,
on different inputs, must each match beam_route given a workspace; sizes past the array's
limit are refused. This file is collected last, so a run that stops at the first failure has
already run everything else."""
import numpy as np
import pytest
import torch

import synth
from synth import BEAM, TINY
from hybrid_attention_moe_gb300 import beam as B

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _route_both(shape, T, seed):
    cfg = B.LayerCfg.from_shape(shape, B.BEAM_ATTN_SWA_ROPE)
    u = synth.activations(T, shape.hidden, seed, "u", DEV)
    R = synth.router_weights(shape, 0, seed, device=DEV)
    ws = torch.empty(B.workspace_bytes(cfg, T, 1), dtype=torch.uint8, device=DEV)
    idx_ref = torch.empty((T, shape.topk), dtype=torch.int32, device=DEV)
    w_ref = torch.empty((T, shape.topk), dtype=torch.float32, device=DEV)
    B.beam_route(cfg, u, R["router"], R["corr_bias"], None, idx_ref, w_ref, ws)
    idx = torch.full_like(idx_ref, -1)
    w = torch.full_like(w_ref, -1.0)
    B.beam_route_noalloc(cfg, u, R["router"], R["corr_bias"], idx, w)
    torch.cuda.synchronize()
    return idx, w, idx_ref, w_ref


@pytest.mark.parametrize("shape,T", [(BEAM, 1), (BEAM, 8), (BEAM, 200), (TINY, 77), (TINY, 256)])
def test_noalloc_route_matches_route_twice(shape, T):
    # two calls in a row: the second must not see anything left by the first
    for seed in (T, T + 1000):
        idx, w, idx_ref, w_ref = _route_both(shape, T, seed)
        assert torch.equal(idx, idx_ref)
        rel = (w - w_ref).abs() / w_ref.abs()
        assert float(rel.max()) <= 1e-5
    assert B.beam_get_device_status() == 0


@pytest.mark.parametrize("shape", [BEAM, TINY])
def test_noalloc_route_rejects_oversize(shape):
    """257 tokens: past the array at 256 experts (257 x 256 > 65536 logits), and past the
    256-token range at 16 experts, where the array would still hold the logits but
    beam_route itself would take its tensor-core form."""
    cfg = B.LayerCfg.from_shape(shape, B.BEAM_ATTN_SWA_ROPE)
    T = 257
    u = torch.zeros((T, shape.hidden), dtype=torch.bfloat16, device=DEV)
    R = synth.router_weights(shape, 0, 0, device=DEV)
    idx = torch.empty((T, shape.topk), dtype=torch.int32, device=DEV)
    w = torch.empty((T, shape.topk), dtype=torch.float32, device=DEV)
    with pytest.raises(B.BeamError, match="invalid argument"):
        B.beam_route_noalloc(cfg, u, R["router"], R["corr_bias"], idx, w)
