"""FP8 e4m3 encoding and the rotate-then-block-quantise step, in float64
(test infrastructure).

"FlashAttention scaling, multi-GPU training and weight quantization" §1
(FlashAttention-3): before the FP8 attention, Q and K are multiplied by a
random orthogonal matrix (incoherent processing) and every small tile is
quantised with its own scale (block quantisation).  The reading used here:
the orthogonal matrix is R = H_D diag(s) / sqrt(D) (Sylvester Hadamard matrix
H_D, signs s = +-1), applied to the rows of each (b, h) matrix; a tile is 128
rows x 128 columns; scale = max |y| / 448 over the tile (1 for an all-zero
tile); code = the e4m3 value nearest to y / scale, ties to even, magnitudes
above 448 held at 448.

The encoder below is written from the OCP E4M3 layout: 3 mantissa bits, so
on [2^e, 2^(e+1)) the representable spacing is 2^(e-3); below 2^-6 the spacing
stays 2^-9 (subnormals); the largest finite value is 448.
"""
from __future__ import annotations

import numpy as np

from .codecs import e4m3_decode

_VALUES = e4m3_decode(np.arange(256, dtype=np.uint8))


def e4m3_encode(x) -> np.ndarray:
    """float64 -> uint8 e4m3 code: nearest representable value, ties to even,
    saturating at +-448.  NaN is not accepted."""
    x = np.asarray(x, dtype=np.float64)
    if np.isnan(x).any():
        raise ValueError("NaN has no saturating e4m3 encoding here")
    a = np.minimum(np.abs(x), 448.0)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.clip(e, -6.0, 8.0)                     # below 2^-6 the spacing stays 2^-9
    quantum = np.exp2(e - 3.0)
    m = a / quantum
    r = np.round(m)                               # numpy rounds half to even
    q = np.minimum(r * quantum, 448.0)
    # map each magnitude to its code (positive codes 0x00..0x7E), then the sign
    pos = _VALUES[:0x7F]
    idx = np.searchsorted(pos, q)
    assert np.array_equal(pos[idx], q), "encoder produced a value e4m3 cannot hold"
    code = idx.astype(np.uint8)
    return np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)   # the sign survives rounding to 0


def hadamard(n: int) -> np.ndarray:
    """Sylvester Hadamard matrix of order n (power of two): H_2n = [[H, H], [H, -H]]."""
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def rotate_quantize(x, signs=None, tile: int = 128):
    """x [B,H,S,D] -> (codes uint8 [B,H,S,D], scales [B,H,ceil(S/tile),ceil(D/tile)],
    y float64 [B,H,S,D]), y = x R (R as above) or x itself when signs is None."""
    x = np.asarray(x, dtype=np.float64)
    B, H, S, D = x.shape
    if signs is not None:
        R = hadamard(D) * np.asarray(signs, dtype=np.float64)[None, :] / np.sqrt(D)
        y = x @ R
    else:
        y = x.copy()
    nts, ntd = -(-S // tile), -(-D // tile)
    scales = np.ones((B, H, nts, ntd))
    codes = np.zeros((B, H, S, D), dtype=np.uint8)
    for ts in range(nts):
        for td in range(ntd):
            blk = y[:, :, ts * tile:(ts + 1) * tile, td * tile:(td + 1) * tile]
            amax = np.abs(blk).max(axis=(2, 3))
            sc = np.where(amax > 0, amax / 448.0, 1.0)
            scales[:, :, ts, td] = sc
            codes[:, :, ts * tile:(ts + 1) * tile, td * tile:(td + 1) * tile] = e4m3_encode(blk / sc[:, :, None, None])
    return codes, scales, y
