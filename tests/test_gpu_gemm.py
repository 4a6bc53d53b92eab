"""The tensor-core GEMM behind the prefill projections, through the C ABI, against a float64
matrix product (NumPy) of the same bf16 inputs: tiles, ragged M/N/K tails, both outputs."""
import numpy as np
import pytest
import torch

import synth
from hybrid_attention_moe_gb300 import beam as B
from parity import np64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (64, 256, 128), (130, 300, 200),
                                   (1000, 1024, 5120), (384, 14336, 5120), (256, 5120, 6144),
                                   (200, 520, 20480)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_gemm_bf16(M, N, K, out):
    a = synth.normal((M, K), 1.0, 0.0, 1, ("gemm_a", M, K), DEV)
    b = synth.normal((N, K), 0.02, 0.0, 1, ("gemm_b", N, K), DEV)
    c = torch.empty((M, N), dtype=torch.float32 if out == "f32" else torch.bfloat16, device=DEV)
    B.beam_gemm_bf16(a, b, c)
    torch.cuda.synchronize()
    ref = np64(a) @ np64(b).T
    got = np64(c)
    scale = np.sqrt(K) * 0.02          # typical |c|
    err = np.abs(got - ref)
    if out == "f32":
        # fp32 accumulation of K exact bf16 products: error ~ sqrt(K) ulps of the partial sums
        assert np.max(err) <= 1e-4 * scale * max(1.0, np.sqrt(K / 1024)), np.max(err)
    else:
        assert np.all(err <= 2 ** -8 * np.abs(ref) + 1e-4 * scale), np.max(err / (np.abs(ref) + scale))


def test_gemm_strided_operands():
    """Row strides larger than K (a view into a wider matrix)."""
    M, N, K = 192, 512, 256
    aw = synth.normal((M, K + 64), 1.0, 0.0, 2, ("wa",), DEV)
    bw = synth.normal((N, K + 128), 0.02, 0.0, 2, ("wb",), DEV)
    a, b = aw[:, :K], bw[:, :K]
    c = torch.empty((M, N), dtype=torch.float32, device=DEV)
    B.beam_gemm_bf16(a, b, c)
    ref = np64(a) @ np64(b).T
    assert np.max(np.abs(np64(c) - ref)) <= 1e-4 * np.sqrt(K) * 0.02
