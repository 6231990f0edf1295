"""Gradients of exact attention, in float64 (test infrastructure).

"Fast Inference and Training at Scale" §6.21 (Idea 2) and "Week 13. GPUs and
FlashAttention" step 2: the backward pass keeps only O and the per-row
log-sum-exp from the forward and recomputes the scores and probabilities.
The gradients themselves follow from the definition O = P V,
P = softmax(S), S = scale * Q K^T (with the mask):

    dV = P^T dO
    dP = dO V^T
    dS = P o (dP - rowsum(dO o O))        (softmax derivative; rowsum(dO o O)
                                           equals rowsum(P o dP))
    dQ = scale * dS K
    dK = scale * dS^T Q

Grouped-query heads: the gradient of a shared key/value head is the sum over
the query heads of its group.  Masked entries have P = 0 and so contribute
nothing; rows with no allowed key have O = 0 and zero gradients.
"""
from __future__ import annotations

import numpy as np

from .attention import attention


def attention_backward(q, k, v, do, causal: bool = False, scale: float | None = None):
    """dQ [B,Hq,Sq,D], dK and dV [B,Hkv,Sk,D] for the loss sum(dO o O)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    g = Hq // Hkv
    O, L = attention(q, k, v, causal, scale)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    rows = np.arange(Sq)[:, None]
    keys = np.arange(Sk)[None, :]
    allowed = (keys <= rows + (Sk - Sq)) if causal else np.ones((Sq, Sk), dtype=bool)
    for b in range(B):
        for h in range(Hq):
            kv = h // g
            s = scale * (q[b, h] @ k[b, kv].T)
            lse = L[b, h][:, None]
            live = np.isfinite(lse)
            P = np.where(allowed & live, np.exp(s - np.where(live, lse, 0.0)), 0.0)  # recomputed from LSE
            dP = do[b, h] @ v[b, kv].T
            Dr = (do[b, h] * O[b, h]).sum(axis=1, keepdims=True)
            dS = P * (dP - Dr)
            dv[b, kv] += P.T @ do[b, h]
            dq[b, h] = scale * dS @ k[b, kv]
            dk[b, kv] += scale * dS.T @ q[b, h]
    return dq, dk, dv, O, L
