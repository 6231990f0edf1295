"""Algorithmic work of each kernel: the numerators of the roofline fractions.

FLOPs count the two matrix products of attention, 2*D per score each
(Q K^T and P V): 4 * B * Hq * Sq * Sk * D, halved under a causal mask (the
keys above the diagonal are never visited -- "Week 13. GPUs and
FlashAttention", step 2).  Bytes are the minimum HBM traffic: every input
read once and every output written once ("Fast Inference and Training at
Scale" §6.21: only O needs to reach HBM).  Decode reads each sequence's
cached K and V once; its intensity is Hq/Hkv FLOP per byte (Week 13 step 1:
"4 for Llama-3-8B, 1 with MHA").
"""
from __future__ import annotations


def prefill_flops(B, Hq, Sq, Sk, D, causal) -> float:
    f = 4.0 * B * Hq * Sq * Sk * D
    return f / 2 if causal else f


def visible_pairs(Sq, Sk, causal) -> int:
    """(query, key) pairs under the mask of one head: all Sq * Sk, or with the
    bottom-right causal alignment, row i sees keys j <= i + Sk - Sq."""
    if not causal:
        return Sq * Sk
    off = Sk - Sq
    return sum(max(0, min(Sk, i + off + 1)) for i in range(Sq))


def prefill_flops_exact(B, Hq, Sq, Sk, D, causal) -> float:
    """4 * D FLOPs per visible (query, key) pair (Q K^T and P V), counted exactly."""
    return 4.0 * D * B * Hq * visible_pairs(Sq, Sk, causal)


def backward_flops(B, Hq, Sq, Sk, D, causal) -> float:
    """Five products per score (S and dP recomputed, dV, dK, dQ), 2*D FLOPs
    each: 2.5 x the forward's count."""
    return 2.5 * prefill_flops(B, Hq, Sq, Sk, D, causal)


def prefill_bytes(B, Hq, Hkv, Sq, Sk, D, elem_bytes=2, out_bytes=2, lse=True) -> float:
    qkv = (B * Hq * Sq * D + 2 * B * Hkv * Sk * D) * elem_bytes
    out = B * Hq * Sq * D * out_bytes + (B * Hq * Sq * 4 if lse else 0)
    return float(qkv + out)


def fp8_scale_bytes(B, Hq, Hkv, Sq, Sk, D, tile=128) -> float:
    t = lambda s: -(-s // tile)  # noqa: E731
    return 4.0 * (B * Hq * t(Sq) * t(D) + 2 * B * Hkv * t(Sk) * t(D))


def decode_kv_bytes(seqlens, Hkv, D, elem_bytes=2) -> float:
    """Bytes of cached K and V that one decode call must read."""
    return float(sum(int(x) for x in seqlens)) * Hkv * D * 2 * elem_bytes


def decode_bytes(seqlens, B, Hq, Hkv, D, elem_bytes=2, lse=True) -> float:
    q_o = 2 * B * Hq * D * elem_bytes + (B * Hq * 4 if lse else 0)
    return decode_kv_bytes(seqlens, Hkv, D, elem_bytes) + q_o + 4 * B


def decode_flops(seqlens, Hq, D) -> float:
    return 4.0 * float(sum(int(x) for x in seqlens)) * Hq * D


def score_matrix_bytes(S, H, elem_bytes=2) -> float:
    """Size of the S x S score matrices of H heads that standard attention
    writes to HBM (and the tiled method never does)."""
    return float(S) * S * H * elem_bytes


def memory_saving_ratio(S, D) -> float:
    """Score matrix (S x S) over output (S x D) per head: S / D."""
    return S / D
