"""The oracle over many (batch, head) pairs at once -- TEST INFRASTRUCTURE ONLY.

Each (b, h) of the attention definition is an independent problem ("Fast
Inference and Training at Scale" §6.21 states it per head; attention.py
computes one head at a time), so whole heads can be handed to separate worker
processes without changing what is computed: every worker calls
``attention`` on a one-head slice exactly as a serial loop would.

The pool uses the "spawn" start method, so it may be created after CUDA has
been initialised in the calling process.  Inputs go to the workers as
memory-mapped .npy files and results come back the same way; each worker keeps
its BLAS library to one thread so the cores are shared by processes, not
oversubscribed.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import tempfile

import numpy as np

_BLAS_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")
_W = {}


def _init(paths, out_paths):
    _W["q"], _W["k"], _W["v"] = (np.load(p, mmap_mode="r") for p in paths)
    _W["o"] = np.load(out_paths[0], mmap_mode="r+")
    _W["l"] = np.load(out_paths[1], mmap_mode="r+")


def _one(task):
    from .attention import attention
    idx, b, h, causal, scale = task
    q, k, v = _W["q"], _W["k"], _W["v"]
    kv = h // (q.shape[1] // k.shape[1])
    O, L = attention(q[b:b + 1, h:h + 1], k[b:b + 1, kv:kv + 1], v[b:b + 1, kv:kv + 1], causal=causal, scale=scale)
    _W["o"][idx] = O[0, 0]
    _W["l"][idx] = L[0, 0]
    _W["o"].flush()
    _W["l"].flush()
    return idx


def default_workers() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def attention_heads(q, k, v, heads, causal: bool, scale: float | None = None, workers: int | None = None):
    """O [len(heads), Sq, D] and LSE [len(heads), Sq] (float64) of the listed
    (b, h) pairs of q [B,Hq,Sq,D] against k/v [B,Hkv,Sk,D] (numpy arrays of any
    float type; they are read as float64 by the definition)."""
    heads = [(int(b), int(h)) for b, h in heads]
    Sq, D = q.shape[2], v.shape[3]
    if scale is None:
        scale = 1.0 / np.sqrt(q.shape[3])
    workers = min(workers or default_workers(), max(1, len(heads)))
    with tempfile.TemporaryDirectory(prefix="oracle_pool_") as d:
        paths = []
        for name, x in (("q", q), ("k", k), ("v", v)):
            p = os.path.join(d, name + ".npy")
            np.save(p, np.ascontiguousarray(x))
            paths.append(p)
        out_paths = (os.path.join(d, "o.npy"), os.path.join(d, "l.npy"))
        np.lib.format.open_memmap(out_paths[0], mode="w+", dtype=np.float64, shape=(len(heads), Sq, D)).flush()
        np.lib.format.open_memmap(out_paths[1], mode="w+", dtype=np.float64, shape=(len(heads), Sq)).flush()
        saved = {n: os.environ.get(n) for n in _BLAS_VARS}
        try:
            for n in _BLAS_VARS:  # the spawned workers read these when their BLAS loads
                os.environ[n] = "1"
            ctx = mp.get_context("spawn")
            with ctx.Pool(workers, initializer=_init, initargs=(paths, out_paths)) as pool:
                done = pool.map(_one, [(i, b, h, bool(causal), float(scale)) for i, (b, h) in enumerate(heads)],
                                chunksize=1)
        finally:
            for n, val in saved.items():
                if val is None:
                    os.environ.pop(n, None)
                else:
                    os.environ[n] = val
        assert sorted(done) == list(range(len(heads)))
        O = np.array(np.load(out_paths[0], mmap_mode="r"))
        L = np.array(np.load(out_paths[1], mmap_mode="r"))
    return O, L
