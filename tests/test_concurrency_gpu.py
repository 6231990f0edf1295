"""Calls from several host threads, each on its own CUDA stream, at once.

The library keeps no per-call state beyond its device error word (and, for
attn_fwd_host, two copy streams and their events per calling thread and
device), and its kernels are deterministic, so calls running concurrently on
different streams must give exactly -- bit for bit -- the results of the
same calls made one at a time."""
import threading

import pytest
import torch

from exact_tiled_attention_15_gb300 import workloads

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def test_threads_on_separate_streams_give_the_serial_results():
    import exact_tiled_attention_15_gb300 as eta
    w1 = workloads.make_prefill(2, 8, 2, 700, 700, 128, seed=61)
    w2 = workloads.make_prefill(1, 4, 4, 1000, 1000, 64, seed=62)
    wd = workloads.make_decode(4, 8, 2, 128, 100, 900, seed=63)
    q1, k1, v1 = (w1[n].to(DEV) for n in ("q", "k", "v"))
    h2 = [w2[n].pin_memory() for n in ("q", "k", "v")]
    qd, kd, vd, sd = (wd[n].to(DEV) for n in ("q", "kcache", "vcache", "seqlens"))
    calls = {
        "device forward (GQA, causal)": lambda: eta.fwd(q1, k1, v1, causal=True),
        "host-buffer forward (D = 64)": lambda: eta.fwd_host(*h2, causal=False, device=DEV),
        "decode": lambda: eta.decode(qd, kd, vd, sd),
    }
    ref = {name: [t.clone() for t in fn()] for name, fn in calls.items()}  # one at a time
    torch.cuda.synchronize()
    assert eta.get_error() == 0

    results, errors = {}, []
    go = threading.Barrier(len(calls))

    def worker(name, fn):
        try:
            stream = torch.cuda.Stream(DEV)
            with torch.cuda.stream(stream):
                go.wait()
                outs = [fn() for _ in range(6)]
            stream.synchronize()
            results[name] = outs
        except Exception as e:  # noqa: BLE001 -- reported below
            errors.append(f"{name}: {e!r}")

    threads = [threading.Thread(target=worker, args=item) for item in calls.items()]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errors, errors
    assert eta.get_error() == 0
    for name, outs in results.items():
        for i, out in enumerate(outs):
            for a, b in zip(out, ref[name]):
                assert torch.equal(a.cpu(), b.cpu()), f"{name}, call {i}: differs from the serial result"
    assert set(results) == set(calls)
