"""The benchmark's multi-rank path (one replica per GPU, no data-path
collective) on CPU with two gloo ranks: the barrier, the max over ranks of the
step time, and the whole-job aggregate."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2",
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    ws, r, local = bench.dist_setup(None)
    step_ms = 2.0 if rank == 0 else 3.0  # rank 1 is the slow one
    bench.barrier(ws)
    m = bench.max_over_ranks(step_ms, ws)
    q.put((r, ws, m, bench.whole_job_tflops(1e12, ws, m)))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_max_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=100) for _ in range(2))
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    for r, ws, m, v in out:
        assert ws == 2
        assert m == 3.0                      # both ranks see the slowest time
        assert v == pytest.approx(2 * 1e12 / 3e-3 / 1e12)  # both replicas' work over that time


def test_single_rank_aggregate():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.25, 1) == 1.25
    assert bench.whole_job_tflops(549.755813888e9, 1, 0.5) == pytest.approx(1099.5, rel=1e-4)


def test_bench_sample_parity_grades_like_the_tests():
    """bench.sample_parity: 1e-2 plus half a bf16 ulp of the oracle's O, and
    1e-3 on the LSE; a kept GPU output is compared head by head."""
    import numpy as np
    import torch
    import bench
    rng = np.random.default_rng(0)
    O = rng.standard_normal((2, 5, 4)) * 3
    L = rng.standard_normal((2, 5))
    L[1, 4] = -np.inf
    o = torch.zeros(1, 3, 5, 4, dtype=torch.float64)
    lse = torch.zeros(1, 3, 5, dtype=torch.float64)
    heads = [(0, 2), (0, 0)]
    for i, (b, h) in enumerate(heads):
        o[b, h] = torch.from_numpy(O[i] + 0.009)
        lse[b, h] = torch.from_numpy(L[i] + 5e-4)
    bench._GPU_OUT["t"] = (o, lse)
    try:
        r = bench.sample_parity("t", heads, O, L)
        assert r["within_bound"] and r["heads"] == 2 and r["elements_over_1e-2"] == 0
        assert abs(r["max_abs_dO"] - 0.009) < 1e-12 and abs(r["max_abs_dLSE"] - 5e-4) < 1e-12
        o[0, 0, 0, 0] += 0.05  # beyond 1e-2 + half an ulp of |O| < 16
        assert not bench.sample_parity("t", heads, O, L)["within_bound"]
        assert bench.sample_parity("absent", heads, O, L) is None
    finally:
        bench._GPU_OUT.pop("t", None)
