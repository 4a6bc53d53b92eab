"""Number formats used at the layer's storage points, written from their definitions.

TEST INFRASTRUCTURE (see oracle/__init__.py): never imported by the product path.

bfloat16: the upper 16 bits of an IEEE-754 binary32 value (1 sign, 8 exponent, 7 fraction
bits); a binary32 value is rounded to it to nearest, ties to even.

FP8 e4m3 ("fn" variant of the OCP 8-bit floating point specification): 1 sign bit, 4 exponent
bits with bias 7, 3 fraction bits; exponent field 0 encodes subnormals m/8 * 2^-6; no
infinities; S.1111.111 is NaN, so the largest finite magnitude is 1.75 * 2^8 = 448.
Encoding here is round-to-nearest-even with saturation to +-448 ("satfinite"), the rule the
Beam page's FP8 KV cache needs (vLLM page, "--kv-cache-dtype fp8"; the quantisation rule
itself is not printed, so saturation is the stated reading).

FP4 e2m1: 1 sign bit, 2 exponent bits with bias 1, 1 fraction bit; exponent field 0 encodes
the subnormal m * 0.5; no infinities or NaN, so the magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6.
NVFP4 (the expert weight format the Beam and Flint pages name for the shipped checkpoints;
the pages do not print its layout, so NVIDIA's published definition is the reading): e2m1
elements in blocks of 16 consecutive elements of a row, each block scaled by one e4m3 value,
and the whole matrix by one FP32 value; element = e2m1 * block scale * matrix scale. Two
elements share a byte, the even element in the low nibble.

Block-scaled FP8 (the FP8 expert weights: the AREX feed article on the Day-0 support says the
weights ship in BF16, FP8 and NVFP4 and prints no FP8 layout; the reading is the block-scaled
e4m3 format of the DeepSeek-V3 release, whose routing the Beam page names): e4m3 codes, one FP32
scale per 128 x 128 block of the [rows][K] matrix (ragged blocks at the edges); element =
e4m3 * scale of its block.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def f32(x) -> np.ndarray:
    """Round to binary32 (numpy's float64 -> float32 cast rounds to nearest even)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def bf16_bits(x) -> np.ndarray:
    """bfloat16 bit patterns (uint16) of x, rounding x to binary32 first, then to nearest-even."""
    f = np.ascontiguousarray(f32(x))
    u = f.view(np.uint32).astype(np.uint64)
    nan = np.isnan(f)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    # a NaN keeps its sign and becomes the quiet NaN pattern
    r = np.where(nan, (u >> np.uint64(16)).astype(np.uint16) | np.uint16(0x0040), r)
    return r


def bf16_from_bits(b) -> np.ndarray:
    u = (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16))
    with np.errstate(invalid="ignore"):
        return np.ascontiguousarray(u).view(np.float32).astype(np.float64)


def bf16_round(x) -> np.ndarray:
    """x rounded to bfloat16, returned as float64 (exactly representable)."""
    return bf16_from_bits(bf16_bits(x))


def e4m3_table() -> np.ndarray:
    """Value of each of the 256 e4m3 codes (float64; NaN for the two NaN codes)."""
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            vals[code] = np.nan
        elif e == 0:
            vals[code] = sign * (m / 8.0) * 2.0 ** -6
        else:
            vals[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_E4M3 = e4m3_table()
# positive finite magnitudes, in code order 0x00..0x7E (increasing)
_E4M3_POS = _E4M3[:0x7F]


def e4m3_decode(codes) -> np.ndarray:
    return _E4M3[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(x) -> np.ndarray:
    """Codes (uint8) of x rounded to nearest-even on the e4m3 grid, saturated to +-448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    with np.errstate(divide="ignore", invalid="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)                 # subnormal binade shares the 2^-6 exponent
    quantum = 2.0 ** (e - 3.0)              # 3 fraction bits
    q = np.rint(a / quantum) * quantum      # rint: ties to even on the integer multiple
    q = np.minimum(q, E4M3_MAX)
    code = np.searchsorted(_E4M3_POS, q).astype(np.uint8)
    code = np.where(np.signbit(x), code | np.uint8(0x80), code)
    code = np.where(np.isnan(x), np.uint8(0x7F), code)
    return code.astype(np.uint8)


def e2m1_table() -> np.ndarray:
    """Value of each of the 16 e2m1 codes (float64)."""
    vals = np.empty(16, dtype=np.float64)
    for code in range(16):
        sign = -1.0 if code & 0x8 else 1.0
        e = (code >> 1) & 0x3
        m = code & 0x1
        vals[code] = sign * (m * 0.5 if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1))
    return vals


_E2M1 = e2m1_table()
NVFP4_BLOCK = 16


def e2m1_decode(codes) -> np.ndarray:
    return _E2M1[np.asarray(codes, dtype=np.uint8) & np.uint8(0xF)]


def nvfp4_unpack(packed) -> np.ndarray:
    """Codes [..., 2n] of packed bytes [..., n]: element 2i is the low nibble of byte i."""
    b = np.asarray(packed, dtype=np.uint8)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = b & np.uint8(0xF)
    out[..., 1::2] = b >> np.uint8(4)
    return out


def nvfp4_dequant(packed, scales, matrix_scale) -> np.ndarray:
    """Values [rows][K] (float64) of an NVFP4 matrix: packed [rows][K/2] bytes, scales
    [rows][K/16] e4m3 codes, one FP32 matrix scale."""
    v = e2m1_decode(nvfp4_unpack(packed))
    s = e4m3_decode(scales)
    rows, K = v.shape
    v = v.reshape(rows, K // NVFP4_BLOCK, NVFP4_BLOCK) * s[:, :, None]
    return v.reshape(rows, K) * float(np.float32(matrix_scale))


FP8_BLOCK = 128


def fp8_block_dequant(codes, scales) -> np.ndarray:
    """Values [rows][K] (float64) of a block-scaled FP8 matrix: codes [rows][K] e4m3 bytes,
    scales [ceil(rows/128)][ceil(K/128)] FP32, one per 128 x 128 block."""
    v = e4m3_decode(codes)
    s = np.asarray(scales, dtype=np.float32).astype(np.float64)
    rows, K = v.shape
    rb = np.arange(rows) // FP8_BLOCK
    kb = np.arange(K) // FP8_BLOCK
    return v * s[rb[:, None], kb[None, :]]
