"""Exact attention by its plain definition, in float64 (test infrastructure).

Follows "Fast Inference and Training at Scale" (§6.21, "Standard Attention"):
form the score matrix S = scale * Q K^T, take a row-wise softmax P, and output
O = P V.  Every row of S is complete before its softmax is taken; nothing is
tiled.  The log-sum-exp of each row (what "Week 13. GPUs and FlashAttention",
step 2, says the forward keeps for the backward pass) is returned beside O.

Readings where the pages are silent:
  * scale defaults to 1/sqrt(D) (the sqrt(d_k) of the §6.21 formula);
  * grouped-query heads (§6.2): query head h reads key/value head
    h // (Hq // Hkv), i.e. contiguous groups;
  * causal mask with Sq != Sk is aligned at the bottom right: key j is allowed
    for query i iff j <= i + (Sk - Sq);
  * a row with no allowed key has O = 0 and LSE = -inf;
  * LSE is the natural log of sum_j exp(s_ij) over the allowed keys, with the
    scale already applied.
"""
from __future__ import annotations

import numpy as np


def _allowed(Sq: int, Sk: int, causal: bool, rows: np.ndarray) -> np.ndarray:
    """Boolean [len(rows), Sk]: which keys each query row may attend to."""
    keys = np.arange(Sk)[None, :]
    if not causal:
        return np.ones((len(rows), Sk), dtype=bool)
    return keys <= (rows[:, None] + (Sk - Sq))


def _softmax_rows(s: np.ndarray, allowed: np.ndarray, v: np.ndarray):
    """Softmax of each (masked) score row, then the weighted sum of V rows.

    s [R, Sk], allowed [R, Sk], v [Sk, D]; returns O [R, D], LSE [R].
    """
    s = np.where(allowed, s, -np.inf)
    m = s.max(axis=1)                              # row maximum (for stability only)
    any_allowed = allowed.any(axis=1)
    m_safe = np.where(any_allowed, m, 0.0)
    p = np.exp(s - m_safe[:, None])                # exp(-inf) = 0 on masked keys
    l = p.sum(axis=1)                              # softmax denominator
    l_safe = np.where(l > 0, l, 1.0)
    P = p / l_safe[:, None]                        # each allowed row sums to 1
    O = P @ v
    lse = np.where(any_allowed, m_safe + np.log(l_safe), -np.inf)
    O[~any_allowed] = 0.0
    return O, lse


def attention_rows(q, k, v, b: int, h: int, rows, causal: bool, scale: float):
    """O and LSE for the selected query rows of one (batch, query head).

    q [B,Hq,Sq,D], k/v [B,Hkv,Sk,D] (any float type, computed in float64).
    Returns O [len(rows), D] and LSE [len(rows)] in float64.
    """
    Hq, Hkv = q.shape[1], k.shape[1]
    Sq, Sk = q.shape[2], k.shape[2]
    kv = h // (Hq // Hkv)
    rows = np.asarray(rows, dtype=np.int64)
    qi = np.asarray(q[b, h], dtype=np.float64)[rows]
    kj = np.asarray(k[b, kv], dtype=np.float64)
    vj = np.asarray(v[b, kv], dtype=np.float64)
    s = scale * (qi @ kj.T)                        # scores of these rows, all keys
    return _softmax_rows(s, _allowed(Sq, Sk, causal, rows), vj)


def attention(q, k, v, causal: bool = False, scale: float | None = None, row_block: int = 1024):
    """Full O [B,Hq,Sq,D] and LSE [B,Hq,Sq] in float64.

    The score matrix of each (b, h) is formed ``row_block`` complete rows at a
    time only to bound memory; each row is still handled in one piece.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Hq, Sq, D = q.shape
    Hkv = k.shape[1]
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    O = np.zeros((B, Hq, Sq, v.shape[-1]))
    L = np.zeros((B, Hq, Sq))
    for b in range(B):
        for h in range(Hq):
            for r0 in range(0, Sq, row_block):
                rows = np.arange(r0, min(Sq, r0 + row_block))
                O[b, h, rows], L[b, h, rows] = attention_rows(q, k, v, b, h, rows, causal, scale)
    return O, L


def decode(q, kcache, vcache, seqlens, scale: float | None = None):
    """One query token per sequence against its cached keys and values.

    "Fast Inference and Training at Scale" §6.1: at step t the new token's query
    attends over every cached position of its sequence (the cache already holds
    the new token's K and V).  q [B,Hq,D], cache [B,Hkv,Lmax,D], seqlens [B]:
    positions j < seqlens[b] are the sequence; later rows are never used.
    Returns O [B,Hq,D] and LSE [B,Hq] in float64.
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Hkv = kcache.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    g = Hq // Hkv
    O = np.zeros((B, Hq, D))
    L = np.zeros((B, Hq))
    for b in range(B):
        n = int(seqlens[b])
        if n <= 0:                                  # empty sequence: no keys
            L[b] = -np.inf
            continue
        for h in range(Hq):
            kv = h // g
            kj = np.asarray(kcache[b, kv, :n], dtype=np.float64)
            vj = np.asarray(vcache[b, kv, :n], dtype=np.float64)
            s = scale * (kj @ q[b, h])[None, :]
            o, l = _softmax_rows(s, np.ones_like(s, dtype=bool), vj)
            O[b, h], L[b, h] = o[0], l[0]
    return O, L


def merge_partials(o_parts, lse_parts):
    """Merge attention results computed over disjoint key subsets.

    o_parts [n, ..., D] are the softmax-normalised outputs of each subset and
    lse_parts [n, ...] their log-sum-exps.  The merged result is what the whole
    key set gives: lse = log sum_s exp(lse_s) and O = sum_s exp(lse_s - lse) O_s.
    This is the running-max/running-sum update of the online softmax
    ("Hardware Co-Design", FlashAttention section) applied to whole subsets.
    Subsets with lse = -inf (no keys) contribute nothing.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = lse_parts.max(axis=0)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    w = np.exp(lse_parts - m_safe)                  # 0 for empty subsets
    tot = w.sum(axis=0)
    tot_safe = np.where(tot > 0, tot, 1.0)
    lse = np.where(tot > 0, m_safe + np.log(tot_safe), -np.inf)
    O = (w[..., None] * o_parts).sum(axis=0) / tot_safe[..., None]
    return O, lse


def decode_paged(q, k_pages, v_pages, block_table, seqlens, page_size: int, scale: float | None = None):
    """Decode against a paged KV cache ("Fast Inference and Training at
    Scale" §6.3, PagedAttention: a sequence's cache lives in fixed-size blocks
    found through its block table).  Position t of sequence b is row
    t % page_size of page block_table[b, t // page_size]; the rows are
    gathered in position order and the result is `decode` on them.
    """
    B, Hq, D = np.asarray(q).shape
    Hkv = k_pages.shape[1]
    Lmax = block_table.shape[1] * page_size
    kc = np.zeros((B, Hkv, Lmax, D))
    vc = np.zeros((B, Hkv, Lmax, D))
    for b in range(B):
        for t in range(int(seqlens[b])):
            page = int(block_table[b, t // page_size])
            kc[b, :, t] = np.asarray(k_pages[page, :, t % page_size], dtype=np.float64)
            vc[b, :, t] = np.asarray(v_pages[page, :, t % page_size], dtype=np.float64)
    return decode(q, kc, vc, seqlens, scale)


def decode_multi(q, kcache, vcache, seqlens, causal: bool = True, scale: float | None = None):
    """T query tokens per sequence against its cache: q [B,Hq,T,D],
    cache [B,Hkv,Lmax,D].  The tokens are the last T positions of the
    sequence (its cache already holds their K and V), so with the causal mask
    token t (position seqlens[b] - T + t) sees keys up to its own position --
    the bottom-right alignment of `attention` with Sq = T, Sk = seqlens[b].
    This is the verification pass of speculative decoding ("Week 13. GPUs and
    FlashAttention", step 1: gamma + 1 tokens per sequence in one pass).
    Returns O [B,Hq,T,D], LSE [B,Hq,T].
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, T, D = q.shape
    O = np.zeros((B, Hq, T, D))
    L = np.full((B, Hq, T), -np.inf)
    for b in range(B):
        n = int(seqlens[b])
        if n <= 0:
            continue
        O[b:b + 1], L[b:b + 1] = attention(q[b:b + 1], np.asarray(kcache[b:b + 1, :, :n], dtype=np.float64),
                                           np.asarray(vcache[b:b + 1, :, :n], dtype=np.float64), causal, scale)
    return O, L
