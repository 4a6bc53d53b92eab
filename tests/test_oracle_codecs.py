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


def test_e2m1_codes_are_the_published_magnitudes():
    # NVIDIA's FP4 e2m1 lists exactly these eight magnitudes; the sign bit negates them
    vals = codecs.e2m1_table()
    assert list(vals[:8]) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert np.array_equal(vals[8:], -vals[:8])
    assert np.signbit(vals[8])   # code 8 is -0


def test_nvfp4_nibble_order_block_and_matrix_scales():
    # one row of 32 elements: byte 0 = 0x21 holds element 0 = code 1 (0.5) in its low nibble
    # and element 1 = code 2 (1.0) in its high nibble; byte 8 = 0xF7 holds element 16 = code 7
    # (6.0) and element 17 = code 15 (-6.0); block 0 is scaled by e4m3 0x38 = 1.0 and block 1 by
    # 0x40 = 2.0; the matrix scale is 0.25
    packed = np.zeros((1, 16), dtype=np.uint8)
    packed[0, 0] = 0x21
    packed[0, 8] = 0xF7
    scales = np.array([[0x38, 0x40]], dtype=np.uint8)
    v = codecs.nvfp4_dequant(packed, scales, 0.25)
    expect = np.zeros((1, 32))
    expect[0, 0], expect[0, 1] = 0.5 * 0.25, 1.0 * 0.25
    expect[0, 16], expect[0, 17] = 6.0 * 2.0 * 0.25, -6.0 * 2.0 * 0.25
    assert np.array_equal(v, expect)


def test_nvfp4_dequant_matches_element_loop():
    rng = np.random.default_rng(3)
    rows, K = 5, 64
    packed = rng.integers(0, 256, size=(rows, K // 2), dtype=np.uint8)
    scales = rng.integers(0x30, 0x40, size=(rows, K // 16), dtype=np.uint8)
    ms = np.float32(0.004)
    got = codecs.nvfp4_dequant(packed, scales, ms)
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for r in range(rows):
        for k in range(K):
            byte = int(packed[r, k // 2])
            code = byte & 0xF if k % 2 == 0 else byte >> 4
            val = (-1.0 if code & 8 else 1.0) * mags[code & 7]
            sc = float(torch.tensor([int(scales[r, k // 16])], dtype=torch.uint8)
                       .view(torch.float8_e4m3fn).float()[0])
            assert got[r, k] == val * sc * float(ms)


def test_fp8_block_scales_hand_built():
    # a 130 x 260 matrix: two row blocks (128 and a ragged 2) and three column blocks (128, 128
    # and a ragged 4); every code is e4m3 0x38 = 1.0, so each element shows its block's scale
    codes = np.full((130, 260), 0x38, dtype=np.uint8)
    scales = np.array([[1.0, 2.0, 3.0], [4.0, 5.0, 6.0]], dtype=np.float32)
    v = codecs.fp8_block_dequant(codes, scales)
    assert v[0, 0] == 1.0 and v[127, 127] == 1.0
    assert v[127, 128] == 2.0 and v[0, 255] == 2.0 and v[0, 256] == 3.0 and v[127, 259] == 3.0
    assert v[128, 0] == 4.0 and v[129, 128] == 5.0 and v[129, 259] == 6.0
    # the code's sign and magnitude carry through: 0xC4 = -(1 + 4/8) * 2^1 = -3
    codes[129, 259] = 0xC4
    assert codecs.fp8_block_dequant(codes, scales)[129, 259] == -18.0


def test_fp8_block_dequant_matches_element_loop():
    rng = np.random.default_rng(4)
    rows, K = 200, 300
    codes = (rng.integers(0, 0x7F, size=(rows, K), dtype=np.uint8)
             | (rng.integers(0, 2, size=(rows, K), dtype=np.uint8) << 7)).astype(np.uint8)
    scales = rng.uniform(0.001, 0.01, size=(2, 3)).astype(np.float32)
    got = codecs.fp8_block_dequant(codes, scales)
    dec = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    for r in range(rows):
        for k in range(K):
            assert got[r, k] == dec[r, k] * float(scales[r // 128, k // 128])
