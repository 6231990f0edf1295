"""Number-format decoders and FP8 tile dequantisation (test infrastructure).

The pages name the formats but print neither bit layout (FP8 for
FlashAttention-3 in "FlashAttention scaling, multi-GPU training and weight
quantization" §1; FP16/BF16 in "Fast Inference and Training at Scale" §6.22).
The decoders below are written from the published layouts:

  bf16:  1 sign, 8 exponent (bias 127), 7 mantissa bits -- the top half of an
         IEEE-754 binary32.
  e4m3:  the OCP 8-bit floating point "E4M3" format: 1 sign, 4 exponent
         (bias 7), 3 mantissa bits; exponent field 0 is subnormal
         (value = m/8 * 2^-6); no infinities; S.1111.111 is NaN; largest
         finite magnitude 1.75 * 2^8 = 448.

Block quantisation (FlashAttention-3's "scaling small tiles independently")
stores one fp32 scale per 128 x 128 tile; the real value is code x scale.
"""
from __future__ import annotations

import numpy as np


def bf16_decode(codes) -> np.ndarray:
    """uint16 bf16 bit patterns -> float64, exactly."""
    c = np.asarray(codes, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):
        return c.view(np.float32).astype(np.float64)


def e4m3_decode(codes) -> np.ndarray:
    """uint8 e4m3 bit patterns -> float64, exactly (NaN for S.1111.111)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    subnormal = (m / 8.0) * 2.0 ** -6
    val = np.where(e == 0, subnormal, normal)
    val = np.where((e == 0xF) & ((c & 0x7) == 0x7), np.nan, val)
    return sign * val


def dequantize_tiles(codes, scales, tile: int = 128) -> np.ndarray:
    """Real values of block-quantised e4m3 data.

    codes uint8 [B,H,S,D]; scales float32 [B,H,ceil(S/tile),ceil(D/tile)].
    Element (b,h,s,d) is e4m3(code) * scales[b,h,s//tile,d//tile].
    """
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.float64)
    B, H, S, D = codes.shape
    si = np.arange(S) // tile
    di = np.arange(D) // tile
    full = scales[:, :, si][:, :, :, di]             # [B,H,S,D] scale of each element
    return e4m3_decode(codes) * full
