"""Pins of the oracle's number formats against torch's dtype conversions (library routines)
and against closed forms of the formats' definitions."""
import numpy as np
import torch

from oracle import codecs


def test_bf16_decode_exhaustive_matches_torch():
    codes = np.arange(1 << 16, dtype=np.uint16)
    ours = codecs.bf16_from_bits(codes)
    ref = torch.from_numpy(codes.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.all(both_nan | (ours == ref))


def test_bf16_encode_random_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(500_000).astype(np.float32),
        (rng.standard_normal(250_000) * 1e30).astype(np.float32),
        (rng.standard_normal(250_000) * 1e-38).astype(np.float32),   # subnormal range
    ])
    ours = codecs.bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_ties_go_to_even():
    # 1 + 2^-8 lies halfway between bf16 neighbours 1 and 1 + 2^-7: ties to the even (1.0)
    assert codecs.bf16_round(1.0 + 2.0 ** -8) == 1.0
    # 1 + 3 * 2^-8 is halfway between 1 + 2^-7 (odd) and 1 + 2^-6 (even)
    assert codecs.bf16_round(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    assert codecs.bf16_round(3.39e38) == np.float32(3.3895313892515355e38)
    assert np.isinf(codecs.bf16_round(3.4028235e38))


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = codecs.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.all(both_nan | (ours == ref))
    assert np.nanmax(ours) == 448.0 and np.sum(np.isnan(ours)) == 2
    assert ours[1] == 2.0 ** -9          # smallest subnormal


def test_e4m3_encode_in_range_matches_torch():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(400_000) * 3.0,
        rng.uniform(-448, 448, 200_000),
        rng.standard_normal(100_000) * 2.0 ** -8,     # subnormals
        codecs.e4m3_table()[np.isfinite(codecs.e4m3_table())],   # exact grid points
    ]).astype(np.float32)
    # midpoints between neighbours exercise ties-to-even
    grid = np.unique(np.abs(codecs.e4m3_table()[np.isfinite(codecs.e4m3_table())]))
    mids = ((grid[1:] + grid[:-1]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids])
    ours = codecs.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_saturates_and_keeps_nan():
    assert codecs.e4m3_decode(codecs.e4m3_encode(np.array([1000.0, -1e9, 464.0])))\
        .tolist() == [448.0, -448.0, 448.0]
    assert codecs.e4m3_encode(np.array([np.nan]))[0] == 0x7F
    # 0.5 * smallest subnormal ties to even: 0
    assert codecs.e4m3_decode(codecs.e4m3_encode(np.array([2.0 ** -10])))[0] == 0.0
