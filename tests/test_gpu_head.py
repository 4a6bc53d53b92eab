"""GPU parity of beam_lm_head (the LM head with the 30*tanh(z/30) logit softcap) against the
oracle on the same seeded inputs: each projection path (one-token SIMT GEMV, the mma.sync
GEMV for 2-64 tokens, the SIMT GEMV when H is not a multiple of 32, the tensor-core GEMM from
64 tokens), ragged vocabularies, saturating logits, no cap, and the full 201,088-row
vocabulary at hidden 5120 on sampled rows.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
import synth
from synth import BEAM
from hybrid_attention_moe_gb300 import beam as B
from parity import assert_logits_close, np64

pytestmark = pytest.mark.gpu
DEV = "cuda"
VOCAB = 201_088


def shape_h(H):
    return dataclasses.replace(BEAM, hidden=H)


def check_status():
    bits = B.beam_get_device_status()
    assert bits == 0, f"device status bits {bits:#x}"


@pytest.mark.parametrize("T,H,V,std,cap", [
    (1, 256, 1000, 0.02, 30.0), (1, 5120, 4113, 1.0, 30.0), (2, 256, 1000, 0.02, 0.0),
    (3, 256, 517, 1.0, 30.0), (5, 264, 300, 0.5, 30.0), (8, 5120, 4113, 0.02, 30.0),
    (64, 256, 517, 0.5, 30.0), (130, 512, 1000, 0.02, 0.0)])
def test_lm_head(T, H, V, std, cap):
    """std 1.0 puts most logits deep in the cap's saturation (|z| ~ 70); 0.0 = no cap."""
    seed = 7 + T
    W = synth.lm_head_weights(shape_h(H), V, seed, device=DEV, std=std)
    u = synth.activations(T, H, seed, "u_final", DEV)
    logits = torch.empty((T, V), dtype=torch.float32, device=DEV)
    B.beam_lm_head(u, W["w_lm"], logits, softcap=cap)
    check_status()
    ref = O.lm_head(np64(u), np64(W["w_lm"]), cap)
    assert_logits_close(logits.cpu().double().numpy(), ref, "lm head logits")
    if cap > 0:
        assert float(logits.abs().max()) <= cap


@pytest.mark.parametrize("T", [1, 8])
def test_lm_head_full_vocab_sampled(T):
    """Hidden 5120 over 201,088 vocabulary rows (2.06 GB of BF16 weights), the decode and
    verify-batch sizes: 384 sampled rows (the first, the last, the rest seeded) against the
    oracle; every logit finite and within the cap."""
    W = synth.lm_head_weights(BEAM, VOCAB, 3, device=DEV)
    u = synth.activations(T, BEAM.hidden, 3, "u_final", DEV)
    logits = torch.empty((T, VOCAB), dtype=torch.float32, device=DEV)
    B.beam_lm_head(u, W["w_lm"], logits, softcap=30.0)
    check_status()
    rows = np.unique(np.concatenate([[0, VOCAB - 1],
                                     np.random.default_rng(5).integers(0, VOCAB, 382)]))
    ref = O.lm_head(np64(u), np64(W["w_lm"][torch.from_numpy(rows).to(DEV)]), 30.0)
    assert_logits_close(logits[:, torch.from_numpy(rows).to(DEV)].cpu().double().numpy(), ref,
                        "lm head logits, sampled rows")
    assert bool(torch.isfinite(logits).all())
    assert float(logits.abs().max()) <= 30.0


def test_lm_head_rejects_bad_arguments():
    u = torch.zeros((2, 260), dtype=torch.bfloat16, device=DEV)   # H not a multiple of 8
    w = torch.zeros((16, 260), dtype=torch.bfloat16, device=DEV)
    out = torch.empty((2, 16), dtype=torch.float32, device=DEV)
    with pytest.raises(B.BeamError):
        B.beam_lm_head(u, w, out)
    u8 = torch.zeros((2, 256), dtype=torch.bfloat16, device=DEV)
    w8 = torch.zeros((16, 256), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(B.BeamError):
        B.beam_lm_head(u8, w8, out, softcap=float("nan"))
