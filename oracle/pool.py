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
import shutil
import tempfile

import numpy as np

_BLAS_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")
_W = {}


def _init(paths):
    _W["q"], _W["k"], _W["v"] = (np.load(p, mmap_mode="r") for p in paths)


def _one(task):
    from .attention import attention
    idx, b, h, causal, scale, out_paths = task
    q, k, v = _W["q"], _W["k"], _W["v"]
    kv = h // (q.shape[1] // k.shape[1])
    O, L = attention(q[b:b + 1, h:h + 1], k[b:b + 1, kv:kv + 1], v[b:b + 1, kv:kv + 1], causal=causal, scale=scale)
    o = np.load(out_paths[0], mmap_mode="r+")
    lse = np.load(out_paths[1], mmap_mode="r+")
    o[idx] = O[0, 0]
    lse[idx] = L[0, 0]
    o.flush()
    lse.flush()
    return idx


def default_workers() -> int:
    return max(1, len(os.sched_getaffinity(0)))


class HeadPool:
    """Worker processes holding q [B,Hq,Sq,D] and k/v [B,Hkv,Sk,D] (numpy
    arrays of any float type, read as float64 by the definition); ``run`` gives
    O [n, Sq, D] and LSE [n, Sq] (float64) of the listed (b, h) pairs."""

    def __init__(self, q, k, v, workers: int | None = None):
        self.workers = workers or default_workers()
        self.shape_q, self.dv = q.shape, v.shape[3]
        self.dir = tempfile.mkdtemp(prefix="oracle_pool_")
        paths = []
        for name, x in (("q", q), ("k", k), ("v", v)):
            p = os.path.join(self.dir, name + ".npy")
            np.save(p, np.ascontiguousarray(x))
            paths.append(p)
        saved = {n: os.environ.get(n) for n in _BLAS_VARS}
        try:
            for n in _BLAS_VARS:  # the spawned workers read these when their BLAS loads
                os.environ[n] = "1"
            self.pool = mp.get_context("spawn").Pool(self.workers, initializer=_init, initargs=(paths,))
        finally:
            for n, val in saved.items():
                if val is None:
                    os.environ.pop(n, None)
                else:
                    os.environ[n] = val

    def run(self, heads, causal: bool, scale: float | None = None):
        heads = [(int(b), int(h)) for b, h in heads]
        Sq = self.shape_q[2]
        if scale is None:
            scale = 1.0 / np.sqrt(self.shape_q[3])
        out_paths = (os.path.join(self.dir, "o.npy"), os.path.join(self.dir, "l.npy"))
        np.lib.format.open_memmap(out_paths[0], mode="w+", dtype=np.float64, shape=(len(heads), Sq, self.dv)).flush()
        np.lib.format.open_memmap(out_paths[1], mode="w+", dtype=np.float64, shape=(len(heads), Sq)).flush()
        tasks = [(i, b, h, bool(causal), float(scale), out_paths) for i, (b, h) in enumerate(heads)]
        done = self.pool.map(_one, tasks, chunksize=1)
        assert sorted(done) == list(range(len(heads)))
        O = np.array(np.load(out_paths[0], mmap_mode="r"))
        L = np.array(np.load(out_paths[1], mmap_mode="r"))
        return O, L

    def close(self):
        self.pool.close()
        self.pool.join()
        shutil.rmtree(self.dir, ignore_errors=True)

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def attention_heads(q, k, v, heads, causal: bool, scale: float | None = None, workers: int | None = None):
    """O [len(heads), Sq, D] and LSE [len(heads), Sq] (float64) of the listed
    (b, h) pairs, computed on a pool of at most ``workers`` processes."""
    workers = min(workers or default_workers(), max(1, len(heads)))
    with HeadPool(q, k, v, workers) as pool:
        return pool.run(heads, causal, scale)


# ---------------------------------------------------------------- backward
# The gradients of one (batch, KV head) unit -- its query-head group with the
# shared K and V -- are an independent problem too: backward.py computes
# them by the definition, and dK, dV sum over the group inside that one call,
# so a unit is never split across workers.
_WB = {}


def _init_bwd(paths):
    _WB["q"], _WB["k"], _WB["v"], _WB["do"] = (np.load(p, mmap_mode="r") for p in paths)


def _one_bwd(task):
    from .backward import attention_backward
    idx, b, kv, causal, scale, out_paths = task
    q, k, v, do = _WB["q"], _WB["k"], _WB["v"], _WB["do"]
    g = q.shape[1] // k.shape[1]
    hs = slice(kv * g, (kv + 1) * g)
    dq, dk, dv, _, _ = attention_backward(q[b:b + 1, hs], k[b:b + 1, kv:kv + 1], v[b:b + 1, kv:kv + 1],
                                          do[b:b + 1, hs], causal=causal, scale=scale)
    for arr, path in zip((dq[0], dk[0, 0], dv[0, 0]), out_paths):
        m = np.load(path, mmap_mode="r+")
        m[idx] = arr
        m.flush()
    return idx


def backward_units(q, k, v, do, units, causal: bool, scale: float | None = None, workers: int | None = None):
    """dQ [n, g, Sq, D], dK [n, Sk, D] and dV [n, Sk, D] (float64) of the
    listed (b, kv head) units, computed on a pool of at most ``workers``
    processes; each worker calls ``attention_backward`` on one unit's slice
    exactly as a serial loop would."""
    units = [(int(b), int(kv)) for b, kv in units]
    workers = min(workers or default_workers(), max(1, len(units)))
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    g = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    tmp = tempfile.mkdtemp(prefix="oracle_pool_bwd_")
    try:
        paths = []
        for name, x in (("q", q), ("k", k), ("v", v), ("do", do)):
            p = os.path.join(tmp, name + ".npy")
            np.save(p, np.ascontiguousarray(x))
            paths.append(p)
        outs = [os.path.join(tmp, n + ".npy") for n in ("dq", "dk", "dv")]
        for path, shape in zip(outs, ((len(units), g, Sq, D), (len(units), Sk, D), (len(units), Sk, v.shape[3]))):
            np.lib.format.open_memmap(path, mode="w+", dtype=np.float64, shape=shape).flush()
        saved = {n: os.environ.get(n) for n in _BLAS_VARS}
        try:
            for n in _BLAS_VARS:
                os.environ[n] = "1"
            pool = mp.get_context("spawn").Pool(workers, initializer=_init_bwd, initargs=(paths,))
        finally:
            for n, val in saved.items():
                if val is None:
                    os.environ.pop(n, None)
                else:
                    os.environ[n] = val
        try:
            tasks = [(i, b, kv, bool(causal), float(scale), outs) for i, (b, kv) in enumerate(units)]
            done = pool.map(_one_bwd, tasks, chunksize=1)
        finally:
            pool.close()
            pool.join()
        assert sorted(done) == list(range(len(units)))
        return tuple(np.array(np.load(p, mmap_mode="r")) for p in outs)
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
