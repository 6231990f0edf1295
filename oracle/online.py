"""Tiled online-softmax attention on the CPU, float64 (test infrastructure).

An independent second statement of the method, used only to pin the plain
definition in attention.py: if both agree for every block size, neither has a
dropped rescale or a wrong index.

Per query row the pass keeps a running maximum m, a running sum l and a
running output o, and walks over the keys one block at a time.  Two forms:

  * "per_step" -- the update printed in "Hardware Co-Design" (FlashAttention
    section): m_new = max(m_old, max(s));
    l_new = e^(m_old - m_new) l_old + sum_j e^(s_j - m_new);
    O_new = (e^(m_old - m_new) l_old O_old + sum_j e^(s_j - m_new) V_j) / l_new.
  * "deferred" -- the form of "Week 13. GPUs and FlashAttention" (step 2) and of
    FlashAttention-2 in "FlashAttention scaling, multi-GPU training and weight
    quantization" (§1): o and the sum are kept unnormalised, multiplied by
    e^(m_old - m_new) when the maximum grows, and divided by the sum once at
    the end.

A fully masked block leaves the state unchanged: with m = -inf the factor
e^(m_old - m_new) is taken as 0 instead of evaluating e^(-inf + inf).
"""
from __future__ import annotations

import numpy as np


def _rescale(m_old, m_new):
    """e^(m_old - m_new), with 0 when m_old is -inf (nothing accumulated yet)."""
    out = np.zeros_like(m_new)
    fin = np.isfinite(m_old)
    out[fin] = np.exp(m_old[fin] - m_new[fin])
    return out


def _one_head(q, k, v, causal, scale, block, form):
    Sq = q.shape[0]
    Sk = k.shape[0]
    rows = np.arange(Sq)
    m = np.full(Sq, -np.inf)
    l = np.zeros(Sq)
    o = np.zeros((Sq, v.shape[1]))
    for j0 in range(0, Sk, block):
        cols = np.arange(j0, min(Sk, j0 + block))
        s = scale * (q @ k[cols].T)
        if causal:
            s = np.where(cols[None, :] <= rows[:, None] + (Sk - Sq), s, -np.inf)
        m_new = np.maximum(m, s.max(axis=1))
        live = np.isfinite(m_new)                  # rows with at least one key so far
        m_use = np.where(live, m_new, 0.0)
        p = np.exp(s - m_use[:, None])             # masked scores give exactly 0
        alpha = _rescale(m, m_use)
        l_new = alpha * l + p.sum(axis=1)
        if form == "per_step":
            l_div = np.where(l_new > 0, l_new, 1.0)
            o = ((alpha * l)[:, None] * o + p @ v[cols]) / l_div[:, None]
        elif form == "deferred":
            o = alpha[:, None] * o + p @ v[cols]
        else:
            raise ValueError(form)
        m, l = np.where(live, m_new, -np.inf), l_new
    has = l > 0
    if form == "deferred":
        o = o / np.where(has, l, 1.0)[:, None]
    o[~has] = 0.0
    lse = np.where(has, m + np.log(np.where(has, l, 1.0)), -np.inf)
    return o, lse


def attention_online(q, k, v, causal=False, scale=None, block=128, form="deferred"):
    """O [B,Hq,Sq,D] and LSE [B,Hq,Sq] by the tiled online softmax, float64.

    Key blocks hold ``block`` keys (the last may be shorter).  Grouped-query
    heads read key/value head h // (Hq // Hkv).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Hq, Sq, D = q.shape
    Hkv = k.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    g = Hq // Hkv
    O = np.zeros((B, Hq, Sq, v.shape[-1]))
    L = np.zeros((B, Hq, Sq))
    for b in range(B):
        for h in range(Hq):
            O[b, h], L[b, h] = _one_head(q[b, h], k[b, h // g], v[b, h // g], causal, scale, block, form)
    return O, L
