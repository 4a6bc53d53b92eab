"""Rounding-order sensitivity of the oracle (TEST INFRASTRUCTURE, see oracle/__init__.py).

Two correct implementations of the layer differ in the order of their FP32 sums, so their
values just before each rounding point differ by a few FP32 ulps; where that flips a bf16
rounding, the next step sees a different input, and across chained steps (attention, residual,
norm, router, experts, the next layer) the difference grows. How much it grows is a property of
the computation, not of either implementation. `perturbed_rounding` measures it: inside the
block, each bf16 and FP32 rounding point of the oracle first multiplies its input by
(1 + rel * N(0,1)), with rel at the scale of FP32 accumulation error.
"""
from __future__ import annotations

import contextlib

import numpy as np

from . import beam_oracle as _bo

FP32_SUM_REL = 5e-7   # ~ 2^-24 * log2(5120): blocked FP32 summation over the hidden width


@contextlib.contextmanager
def perturbed_rounding(rel: float = FP32_SUM_REL, seed: int = 0):
    rng = np.random.default_rng(seed)
    orig_bf, orig_f32 = _bo.bf16_round, _bo.f32

    def bf(x):
        x = np.asarray(x, dtype=np.float64)
        return orig_bf(x * (1.0 + rel * rng.standard_normal(x.shape)))

    def f32(x):
        x = np.asarray(x, dtype=np.float64)
        return orig_f32(x * (1.0 + rel * rng.standard_normal(x.shape)))

    _bo.bf16_round, _bo.f32 = bf, f32
    try:
        yield
    finally:
        _bo.bf16_round, _bo.f32 = orig_bf, orig_f32
