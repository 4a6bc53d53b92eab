"""Seeded synthetic inputs shared by the CUDA path's tests, the bench and the oracle's tests.

This package draws random numbers and names layer shapes. It holds none of the layer's
arithmetic, so that both sides of every parity test can be fed from it.
"""
from .beam_inputs import (  # noqa: F401
    BeamShape, TINY, BEAM, derived_seed, normal, uniform_codes, layer_weights, expert_weights,
    expert_weights_nvfp4, expert_weights_fp8, lm_head_weights,
    attention_weights, router_weights, dense_weights,
    activations, kv_cache, decode_positions, prefill_positions,
)
from .tie_free import MIN_GAP, STACK_MIN_GAP, TINY_STACK_MIN_GAP, first_accepted  # noqa: F401
