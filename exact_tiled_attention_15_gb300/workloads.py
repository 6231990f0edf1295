"""Seeded synthetic inputs for the attention kernels and for the CPU oracle.

This module only draws inputs: it holds none of the method's arithmetic (no
attention, no rotation, no quantisation).  Both the CUDA path and the oracle
receive exactly the tensors made here.  Rounding to bf16 uses PyTorch's CPU
cast (round to nearest even).

Recipe (every workload, seed 0 unless the caller passes another seed):
  * generator: NumPy ``default_rng(seed)`` (PCG64);
  * draw order: decode sequence lengths (``integers(Lmin, Lmax + 1, B)``),
    then Q, K, V as float32 ``standard_normal``, then outlier masks (one
    ``random()`` draw per entry, outlier where < fraction), then rotation signs;
  * outliers multiply single entries of the float32 draws before rounding;
  * values are rounded to bf16 once.

Workload shapes follow the attention problem statement of "Fast Inference and
Training at Scale" §6.21 (Q, K, V of N x d_k per head) with grouped-query heads
as in its §6.2 (h query heads, G key/value heads, h/G per group).
"""
from __future__ import annotations

import numpy as np
import torch

# Named workloads.  ``S`` is Sq = Sk for prefill.
WORKLOADS = {
    "tiny": dict(kind="prefill", B=1, Hq=2, Hkv=2, S=128, D=64, causal=None),
    "train_prefill_mha": dict(kind="prefill", B=4, Hq=32, Hkv=32, S=4096, D=128, causal=True),
    "long_gqa_prefill": dict(kind="prefill", B=1, Hq=32, Hkv=8, S=16384, D=128, causal=True,
                             k_outlier_frac=0.01, k_outlier_mult=20.0),
    # a 512-token chunk of new queries against a cache of 8192 keys that already holds them
    "chunked_prefill": dict(kind="chunked_prefill", B=8, Hq=32, Hkv=8, Sq=512, Sk=8192, D=128, causal=True),
    "gqa_decode": dict(kind="decode", B=64, Hq=32, Hkv=8, D=128, Lmin=1024, Lmax=8192),
    "gqa_decode_paged": dict(kind="paged_decode", B=64, Hq=32, Hkv=8, D=128, Lmin=1024, Lmax=8192, page_size=64),
    "fp8_prefill": dict(kind="fp8", B=2, Hq=16, Hkv=16, S=8192, D=128, causal=False,
                        outlier_frac=0.005, outlier_mult=50.0),
}


def to_bf16(x: np.ndarray) -> torch.Tensor:
    """Round a float32 array to bf16 (RNE) with PyTorch's CPU cast."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def _apply_outliers(rng, x: np.ndarray, frac: float, mult: float) -> None:
    mask = rng.random(x.shape, dtype=np.float32) < frac
    x[mask] *= mult


def make_prefill(B, Hq, Hkv, Sq, Sk, D, seed=0, k_outlier_frac=0.0, k_outlier_mult=1.0):
    """bf16 Q [B,Hq,Sq,D], K and V [B,Hkv,Sk,D], entries N(0,1).

    With ``k_outlier_frac`` > 0, that fraction of K's entries (i.i.d. per entry)
    is multiplied by ``k_outlier_mult`` before rounding.
    """
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hq, Sq, D), dtype=np.float32)
    k = rng.standard_normal((B, Hkv, Sk, D), dtype=np.float32)
    v = rng.standard_normal((B, Hkv, Sk, D), dtype=np.float32)
    if k_outlier_frac > 0:
        _apply_outliers(rng, k, k_outlier_frac, k_outlier_mult)
    return dict(q=to_bf16(q), k=to_bf16(k), v=to_bf16(v))


def make_decode(B, Hq, Hkv, D, Lmin, Lmax, seed=0, poison_tail=True, seqlens=None, T=None):
    """One query token per sequence against a contiguous per-sequence KV cache.

    Returns q [B,Hq,D] bf16, kcache/vcache [B,Hkv,Lmax,D] bf16 and seqlens [B]
    int32 drawn uniformly in [Lmin, Lmax] (or the given ``seqlens``, in which
    case that draw is still made so the rest of the stream is unchanged).
    Only the live cache rows (position < seqlens[b]) are drawn: first all of
    K's, in (b, head, position, d) order, then all of V's.  Rows at or beyond a
    sequence's length are NaN when ``poison_tail`` (so any read of them shows
    up in the output), else 0.  With T, q holds T query tokens per sequence:
    [B, Hq, T, D].
    """
    rng = np.random.default_rng(seed)
    drawn = rng.integers(Lmin, Lmax + 1, size=B).astype(np.int32)
    seqlens = drawn if seqlens is None else np.asarray(seqlens, dtype=np.int32)
    q = rng.standard_normal((B, Hq, D) if T is None else (B, Hq, T, D), dtype=np.float32)
    fill = np.nan if poison_tail else 0.0
    caches = []
    for _ in range(2):  # K, then V
        c = torch.full((B, Hkv, Lmax, D), fill, dtype=torch.bfloat16)
        live = rng.standard_normal(int(seqlens.sum()) * Hkv * D, dtype=np.float32)
        off = 0
        for b in range(B):
            n = int(seqlens[b]) * Hkv * D
            c[b, :, :seqlens[b]] = to_bf16(live[off:off + n].reshape(Hkv, int(seqlens[b]), D))
            off += n
        caches.append(c)
    return dict(q=to_bf16(q), kcache=caches[0], vcache=caches[1], seqlens=torch.from_numpy(seqlens))


def make_paged_decode(B, Hq, Hkv, D, Lmin, Lmax, page_size, seed=0, poison=True, seqlens=None, spare_pages=3):
    """The decode workload of make_decode, stored in a paged KV cache.

    K and V rows of sequence b, position t live in page block_table[b, t //
    page_size] at row t % page_size of a shared pool [num_pages, Hkv,
    page_size, D].  Pages are handed out in a seeded random order; unused
    rows (and table entries past a sequence's last page, which point at
    page 0) hold NaN when ``poison``.  Returns q, k_pages, v_pages,
    block_table [B, ceil(Lmax / page_size)] int32, seqlens, and the
    contiguous kcache/vcache the pages were filled from.
    """
    w = make_decode(B, Hq, Hkv, D, Lmin, Lmax, seed=seed, poison_tail=poison, seqlens=seqlens)
    sl = w["seqlens"].numpy()
    max_blocks = -(-Lmax // page_size)
    need = [-(-int(n) // page_size) for n in sl]
    num_pages = sum(need) + spare_pages
    order = np.random.default_rng(seed + 1).permutation(num_pages)
    fill = float("nan") if poison else 0.0
    kp = torch.full((num_pages, Hkv, page_size, D), fill, dtype=torch.bfloat16)
    vp = torch.full((num_pages, Hkv, page_size, D), fill, dtype=torch.bfloat16)
    table = np.zeros((B, max_blocks), dtype=np.int32)
    nxt = 0
    for b in range(B):
        for blk in range(need[b]):
            pid = int(order[nxt])
            nxt += 1
            table[b, blk] = pid
            r0, r1 = blk * page_size, min(int(sl[b]), (blk + 1) * page_size)
            kp[pid, :, :r1 - r0] = w["kcache"][b, :, r0:r1]
            vp[pid, :, :r1 - r0] = w["vcache"][b, :, r0:r1]
    return dict(q=w["q"], k_pages=kp, v_pages=vp, block_table=torch.from_numpy(table), seqlens=w["seqlens"],
                kcache=w["kcache"], vcache=w["vcache"], page_size=page_size)


def make_fp8_prefill(B, Hq, Hkv, Sq, Sk, D, seed=0, outlier_frac=0.005, outlier_mult=50.0):
    """The draws behind the FP8 e4m3 prefill inputs.

    bf16 N(0,1) draws for Q, K, V with ``outlier_frac`` of the entries of each
    multiplied by ``outlier_mult`` (before the bf16 rounding), then D random
    signs (+-1, float64) for the rotation R = H_D diag(signs) / sqrt(D).  The
    e4m3 codes and their one-fp32-scale-per-128x128-tile come from these by the
    rotate + quantise step (Q and K rotated by the same R, V not): the library's
    ``rotate_quantize_fp8_many`` kernel, or the CPU oracle's
    ``rotate_quantize`` where a test needs inputs independent of the GPU.
    """
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hq, Sq, D), dtype=np.float32)
    k = rng.standard_normal((B, Hkv, Sk, D), dtype=np.float32)
    v = rng.standard_normal((B, Hkv, Sk, D), dtype=np.float32)
    for x in (q, k, v):
        _apply_outliers(rng, x, outlier_frac, outlier_mult)
    signs = rng.integers(0, 2, size=D).astype(np.float64) * 2.0 - 1.0
    return dict(q=to_bf16(q), k=to_bf16(k), v=to_bf16(v), signs=signs)


def make_workload(name: str, seed: int = 0, **override):
    """Inputs for a named workload (see ``WORKLOADS``)."""
    cfg = dict(WORKLOADS[name])
    cfg.update(override)
    kind = cfg["kind"]
    if kind == "prefill":
        return make_prefill(cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["S"], cfg["S"], cfg["D"], seed,
                            cfg.get("k_outlier_frac", 0.0), cfg.get("k_outlier_mult", 1.0))
    if kind == "chunked_prefill":
        return make_prefill(cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["Sq"], cfg["Sk"], cfg["D"], seed)
    if kind == "decode":
        return make_decode(cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["Lmin"], cfg["Lmax"], seed)
    if kind == "fp8":
        return make_fp8_prefill(cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["S"], cfg["S"], cfg["D"], seed,
                                cfg["outlier_frac"], cfg["outlier_mult"])
    raise ValueError(kind)
