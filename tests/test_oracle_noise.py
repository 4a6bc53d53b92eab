"""The rounding-order probe behind the chained-step tolerances (oracle/noise.py): inside the
block every bf16 / FP32 rounding point of the oracle sees its input nudged at FP32-sum level,
so a single step moves by at most one bf16 unit in the last place (only near-ties flip);
outside it, and after an exception inside it, the oracle is exactly as before."""
import numpy as np
import pytest

import oracle as O
from oracle import beam_oracle as bo
from oracle.noise import perturbed_rounding


def test_single_step_moves_by_at_most_one_bf16_ulp():
    r = np.random.default_rng(0)
    x = r.standard_normal((64, 1024))
    w = 1 + 0.1 * r.standard_normal(1024)
    base = O.boundary_norm(None, x, None, w, 1, 1e-6)[1]
    with perturbed_rounding(seed=3):
        alt = O.boundary_norm(None, x, None, w, 1, 1e-6)[1]
    ulp = 2.0 ** (np.floor(np.log2(np.abs(base))) - 7)
    assert np.all(np.abs(alt - base) <= ulp)
    frac = np.mean(alt != base)
    assert 0 < frac < 0.01          # the probe is active, and only near-ties flip


def test_oracle_restored_after_the_block():
    orig = (bo.bf16_round, bo.f32)
    with pytest.raises(RuntimeError):
        with perturbed_rounding(seed=1):
            assert bo.bf16_round is not orig[0]
            raise RuntimeError("inside")
    assert (bo.bf16_round, bo.f32) == orig
    x = np.random.default_rng(2).standard_normal((8, 256))
    a = O.rmsnorm(x, np.ones(256), 1e-6)
    assert np.array_equal(bo.bf16_round(a), O.codecs.bf16_round(a))
