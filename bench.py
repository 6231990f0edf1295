#!/usr/bin/env python
"""Benchmark of the exact tiled attention kernels on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  The headline step is one bf16 causal prefill
forward of the training workload (B=4, Hq=Hkv=32, Sq=Sk=4096, D=128, O bf16 +
LSE fp32) on synthetic N(0,1) inputs; ``value`` is attention TFLOP/s
(4*B*Hq*S^2*D, halved for causal), whole job over all ranks.  The same line
carries the other workloads measured the same way (long-context GQA prefill,
GQA decode KV-read GB/s, FP8 prefill TFLOP/s), each with its roofline
fraction, plus the end-to-end figure through the public API with host
buffers (with whether its output equals the device-resident call's, bit for
bit), and the CPU fp64 oracle timed on a bounded sample as a baseline; that
sample's oracle outputs are also compared with the headline's GPU output on
the same heads (``cpu_baseline.parity``).

Timing: W warm-up steps, then K steps each bracketed by CUDA events on the
launching stream, L2 flushed between steps outside the events (a 256 MB write,
then a 256 MB read of another buffer, so that the timed step starts with a
clean L2 that holds none of its inputs and does not pay for writing back the
flush's own dirty lines);
a barrier and a device synchronise bracket the whole timed region; the
maximum over ranks is reported.  SM clocks are sampled with nvidia-smi while
the GPU work runs.  With N > 1 (torchrun) every rank runs its own replica of
the workload (weak scaling; no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = "train_prefill_mha"
# the headline metric, worded as the benchmark this measures names it
HEADLINE_METRIC = "attention TFLOP/s (prefill) & KV-read GB/s (decode), 1\u00d7GB300, % of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}
FP8_OVER_BF16 = 2.0  # nominal dense FP8 / BF16 tensor throughput (4.5 / 2.25 PFLOP/s)


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true", help="only the headline workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--only", choices=["train_prefill_mha", "train_prefill_mha_backward", "long_gqa_prefill", "chunked_prefill",
                                       "gqa_decode", "gqa_decode_paged",
                                       "gqa_decode_T4", "fp8_rotate_quantize", "fp8_prefill"],
                    help="run one workload leg alone and print its figures (for profiling)")
    return ap.parse_args()


# ---------------------------------------------------------------- environment
def dist_setup(args):
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step: float, world_size: int, step_ms_max: float) -> float:
    """Work of all replicas over the slowest rank's step time, in TFLOP/s."""
    return flops_per_step * world_size / (step_ms_max * 1e-3) / 1e12


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return dict(FALLBACK_PEAKS)


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        if self.proc is None:
            return out
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 10:
                rows.append(f)
        os.unlink(self.path)
        if not rows:
            return out
        busy = [r for r in rows if r[4].isdigit() and int(r[4]) > 0] or rows
        mhz = [float(r[1]) for r in busy if r[1].replace(".", "").isdigit()]
        out["sm_mhz"] = statistics.median(mhz) if mhz else None
        out["sm_max_mhz"] = float(rows[0][2]) if rows[0][2].replace(".", "").isdigit() else None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in busy:
            for n, v in zip(names, r[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        out["reasons"] = sorted(reasons)
        out["samples"] = len(busy)
        return out


class NvmlClockSampler:
    """SM clock and clock-event reasons read through NVML (read-only queries)
    every ~1 ms on a host thread, so that even a leg whose timed steps last a
    few milliseconds gets samples of its own.  Unavailable without the NVML
    library; then every query returns None and the nvidia-smi sampler stands."""
    # clock-event reason bits (nvml.h): the ones a timing must be rejected or noted for
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int):
        import ctypes
        import threading
        self.samples = []  # (perf_counter, sm_mhz, reasons bitmask)
        self.ok = False
        self._stop = threading.Event()
        self._thread = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            bus = self._pci_bus_id(device_index)
            if bus is None or nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
                if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(device_index), ctypes.byref(h)) != 0:
                    return
            self._nv, self._h, self._ct = nv, h, ctypes
            fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self._reasons_fn = fn
            self.sm_max = self._query(nv.nvmlDeviceGetMaxClockInfo)
            self.ok = self._query(nv.nvmlDeviceGetClockInfo) is not None
        except Exception:
            self.ok = False

    @staticmethod
    def _pci_bus_id(device_index):
        try:
            import torch
            pr = torch.cuda.get_device_properties(device_index)
            return "%08x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
        except Exception:
            return None

    def _query(self, fn):
        v = self._ct.c_uint()
        return v.value if fn(self._h, self._ct.c_int(1), self._ct.byref(v)) == 0 else None  # 1 = SM clock

    def _loop(self):
        ct = self._ct
        r = ct.c_ulonglong()
        while not self._stop.is_set():
            mhz = self._query(self._nv.nvmlDeviceGetClockInfo)
            reasons = r.value if self._reasons_fn(self._h, ct.byref(r)) == 0 else 0
            self.samples.append((time.perf_counter(), mhz, reasons))
            time.sleep(0.001)

    def start(self):
        if self.ok:
            import threading
            self._thread = threading.Thread(target=self._loop, daemon=True)
            self._thread.start()

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=2)

    def window(self, t0, t1):
        """Median SM MHz, sample count and active reasons inside [t0, t1]."""
        sel = [(m, r) for t, m, r in self.samples if t0 <= t <= t1 and m is not None]
        if not sel:
            return {"sm_mhz": None, "samples": 0, "reasons": []}
        reasons = sorted({name for _, r in sel for bit, name in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(m for m, _ in sel), "samples": len(sel), "reasons": reasons}


# timed windows of the legs (perf_counter seconds), for binning clock samples
LEG_WINDOWS = {}


def source_digest(*names) -> str:
    h = hashlib.sha256()
    for n in names:
        h.update(open(os.path.join(ROOT, "exact_tiled_attention_15_gb300", "csrc", n), "rb").read())
    return h.hexdigest()[:16]


def dram_traffic(kernel: str, workload: str, digest: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken
    on the current source of that kernel (else None)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    for line in open(p):
        f = line.split()
        if len(f) == 4 and not line.startswith("#") and f[0] == kernel and f[1] == workload and f[2] == digest:
            return float(f[3])
    return None


# ---------------------------------------------------------------- timing core
class L2Flush:
    """Between timed steps: write 256 MB (> the 129 MB L2), evicting every input
    of the previous step, then read another 256 MB buffer, so that the dirty
    lines of that write are written back here rather than inside the next timed
    step.  The step then starts with a clean L2 holding none of its inputs."""

    def __init__(self):
        import torch
        n = 64 * 1024 * 1024  # fp32 elements: 256 MB
        self.w = torch.empty(n, dtype=torch.float32, device="cuda")
        self.r = torch.zeros(n, dtype=torch.float32, device="cuda")
        self.out = torch.empty((), dtype=torch.float32, device="cuda")

    def __call__(self):
        import torch
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.out)


def time_steps(fn, steps, warmup, flush, leg=None):
    """Per-step device time (ms) of fn() on the current stream, L2 flushed
    between steps.  With ``leg``, the host-clock window of the timed steps is
    kept in LEG_WINDOWS[leg] (for the clock samples)."""
    import torch
    st = torch.cuda.current_stream()
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    t0 = time.perf_counter()
    for a, b in evs:
        flush()
        a.record(st)
        fn()
        b.record(st)
    torch.cuda.synchronize()
    if leg is not None:
        LEG_WINDOWS[leg] = (t0, time.perf_counter())
    return [a.elapsed_time(b) for a, b in evs]


# ---------------------------------------------------------------- workloads
# two-sided 95 % Student-t quantiles by degrees of freedom (larger: the normal 1.96)
_T95 = {1: 12.706, 2: 4.303, 3: 3.182, 4: 2.776, 5: 2.571, 6: 2.447, 7: 2.365, 8: 2.306, 9: 2.262, 10: 2.228,
        12: 2.179, 15: 2.131, 20: 2.086, 25: 2.060, 30: 2.042, 40: 2.021, 60: 2.000, 120: 1.980}


# Nominal dense per-GPU figures of the datasheet, beside the measured peaks the
# fractions are graded on: bf16 2.25 PFLOP/s, FP8 4.5 PFLOP/s, HBM3e 7.9 TB/s.
SPEC = {"bf16": 2250.0, "fp8": 4500.0, "hbm": 7900.0}


def add_spec(roofline):
    """Add the fraction of the nominal datasheet peak to a roofline object."""
    if not roofline or roofline.get("achieved") is None:
        return roofline
    if roofline["unit"] == "GB/s":
        peak = SPEC["hbm"]
    else:
        peak = SPEC["fp8"] if "Fp8" in roofline.get("kernel", "") else SPEC["bf16"]
    roofline["spec_peak"] = peak
    roofline["frac_of_spec"] = roofline["achieved"] / peak
    roofline["spec_source"] = "nominal datasheet, dense"
    return roofline


def timing_stats(ts):
    """Median, 95th percentile and the half-width of the Student-t 95 %
    confidence interval of the mean, in ms, of per-step times."""
    n = len(ts)
    srt = sorted(ts)
    p95 = srt[min(n - 1, int(round(0.95 * (n - 1))))]
    ci = None
    if n > 1:
        dof = n - 1
        t = next((v for k, v in sorted(_T95.items()) if k >= dof), 1.96)
        ci = t * statistics.stdev(ts) / math.sqrt(n)
    return {"ms_median": statistics.median(ts), "ms_p95": p95, "ms_ci95": ci}


def run_prefill(name, steps, warmup, flush, peaks, e2e_steps=0, leg="same"):
    import torch
    import exact_tiled_attention_15_gb300 as eta
    from exact_tiled_attention_15_gb300 import accounting as acc, workloads
    cfg = workloads.WORKLOADS[name]
    B, Hq, Hkv, S, D, causal = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["S"], cfg["D"], cfg["causal"]
    w = workloads.make_workload(name, seed=0)
    dev = torch.device("cuda")
    q, k, v = (w[n].to(dev) for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, S, device=dev, dtype=torch.float32)
    fn = lambda: eta.fwd(q, k, v, causal=causal, out=o, lse_out=lse)  # noqa: E731
    ts = time_steps(fn, steps, warmup, flush, leg=name if leg == "same" else leg)
    if eta.get_error() != 0:
        raise RuntimeError(f"{name}: device-side error")
    if name == HEADLINE:  # for the parity of the CPU baseline's sample
        _GPU_OUT[name] = (o.cpu(), lse.cpu())
    flops = acc.prefill_flops(B, Hq, S, S, D, causal)
    ms = statistics.mean(ts)
    ach = flops / (ms * 1e-3) / 1e12
    digest = source_digest("fwd_kernel.cuh", "fwd_bf16.cu", "ptx.cuh")
    res = {
        "metric": "attention TFLOP/s (bf16 prefill)", "unit": "TFLOP/s", "value": ach,
        "ms_per_step": ms, **timing_stats(ts), "steps": len(ts),
        "config": {"workload": name, "B": B, "Hq": Hq, "Hkv": Hkv, "Sq": S, "Sk": S, "D": D, "causal": causal},
        "flops_per_step": flops,
        "roofline": {"bound": "tensor", "kernel": "fwd_kernel<Bf16,128>", "achieved": ach, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"],
                     "peak_source": peaks["source"] + " bf16 burst",
                     "traffic": dram_traffic("fwd_kernel<Bf16,128>", name, digest),
                     "algorithmic_bytes": acc.prefill_bytes(B, Hq, Hkv, S, S, D)},
        "gpu_launches": len(ts),
    }
    if e2e_steps > 0:
        # the host-buffer entry (attn_fwd_host): inputs in pinned host memory, outputs read back to
        # pinned host memory, copies and kernels overlapped chunk by chunk inside the call
        hq_, hk_, hv_ = (w[n].pin_memory() for n in ("q", "k", "v"))
        ho = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
        hl = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
        ws = torch.empty(eta.fwd_host_workspace_bytes(B, Hq, Hkv, S, S, D), dtype=torch.uint8, device=dev)

        def e2e():
            eta.fwd_host(hq_, hk_, hv_, causal=causal, out=ho, lse_out=hl, workspace=ws, device=dev)

        te = time_steps(e2e, e2e_steps, 2, flush, leg="e2e")
        em = statistics.mean(te)
        res["e2e"] = {"value": flops / (em * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": em,
                      "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in (q, k, v)),
                      "d2h_bytes_per_step": o.numel() * o.element_size() + lse.numel() * 4, "steps": len(te),
                      "api": "exact_tiled_attention_15_gb300.fwd_host (attn_fwd_host) on pinned host buffers"}
        if name in _GPU_OUT:  # the same result as the device-resident call, bit for bit
            res["e2e"]["equals_device_output"] = bool(torch.equal(ho, _GPU_OUT[name][0]) and
                                                      torch.equal(hl, _GPU_OUT[name][1]))
        del ws
    del q, k, v, o, lse
    return res


def run_chunked_prefill(steps, warmup, flush, peaks):
    """A chunk of new queries against a dense KV cache that already holds them
    (Sq < Sk, causal aligned at the bottom right): attn_fwd with Sq != Sk."""
    import torch
    import exact_tiled_attention_15_gb300 as eta
    from exact_tiled_attention_15_gb300 import accounting as acc, workloads
    name = "chunked_prefill"
    cfg = workloads.WORKLOADS[name]
    B, Hq, Hkv, Sq, Sk, D = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["Sq"], cfg["Sk"], cfg["D"]
    w = workloads.make_workload(name, seed=0)
    dev = torch.device("cuda")
    q, k, v = (w[n].to(dev) for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, Sq, device=dev, dtype=torch.float32)
    fn = lambda: eta.fwd(q, k, v, causal=True, out=o, lse_out=lse)  # noqa: E731
    ts = time_steps(fn, steps, warmup, flush, leg=name)
    if eta.get_error() != 0:
        raise RuntimeError(f"{name}: device-side error")
    flops = acc.prefill_flops_exact(B, Hq, Sq, Sk, D, True)
    ms = statistics.mean(ts)
    ach = flops / (ms * 1e-3) / 1e12
    return {
        "metric": "attention TFLOP/s (bf16 chunked prefill against a KV cache, exact visible pairs)",
        "unit": "TFLOP/s", "value": ach, "ms_per_step": ms, **timing_stats(ts), "steps": len(ts),
        "config": {"workload": name, "B": B, "Hq": Hq, "Hkv": Hkv, "Sq": Sq, "Sk": Sk, "D": D, "causal": True},
        "roofline": {"bound": "tensor", "kernel": "fwd_kernel<Bf16,128>", "achieved": ach,
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"],
                     "peak_source": peaks["source"] + " bf16 burst",
                     "traffic": dram_traffic("fwd_kernel<Bf16,128>", name,
                                             source_digest("fwd_kernel.cuh", "fwd_bf16.cu", "ptx.cuh")),
                     "algorithmic_flops": flops, "algorithmic_bytes": acc.prefill_bytes(B, Hq, Hkv, Sq, Sk, D)},
        "gpu_launches": len(ts),
    }


def run_backward(steps, warmup, flush, peaks):
    """Gradients of the headline causal prefill (dQ, dK, dV from Q, K, V, O,
    LSE and a random dO)."""
    import numpy as np
    import torch
    import exact_tiled_attention_15_gb300 as eta
    from exact_tiled_attention_15_gb300 import accounting as acc, workloads
    name = HEADLINE
    cfg = workloads.WORKLOADS[name]
    B, Hq, Hkv, S, D, causal = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["S"], cfg["D"], cfg["causal"]
    w = workloads.make_workload(name, seed=0)
    dev = torch.device("cuda")
    q, k, v = (w[n].to(dev) for n in ("q", "k", "v"))
    do = workloads.to_bf16(np.random.default_rng(7).standard_normal((B, Hq, S, D)).astype(np.float32)).to(dev)
    o, lse = eta.fwd(q, k, v, causal=causal)
    ws = torch.empty(int(eta.lib().attn_bwd_workspace_bytes(B, Hq, S, D)), dtype=torch.uint8, device=dev)
    fn = lambda: eta.bwd(q, k, v, o, lse, do, causal=causal, workspace=ws)  # noqa: E731
    ts = time_steps(fn, steps, warmup, flush, leg=name + "_backward")
    if eta.get_error() != 0:
        raise RuntimeError("backward: device-side error")
    flops = acc.backward_flops(B, Hq, S, S, D, causal)
    ms = statistics.mean(ts)
    ach = flops / (ms * 1e-3) / 1e12
    return {
        "metric": "attention backward TFLOP/s (bf16, recomputation)", "unit": "TFLOP/s", "value": ach,
        "ms_per_step": ms, **timing_stats(ts), "steps": len(ts),
        "config": {"workload": name + "_backward", "B": B, "Hq": Hq, "Hkv": Hkv, "Sq": S, "Sk": S, "D": D,
                   "causal": causal},
        "roofline": {"bound": "tensor", "kernel": "bwd_pre + bwd_kernel<128> + bwd_post", "achieved": ach,
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"],
                     "peak_source": peaks["source"] + " bf16 burst",
                     "traffic": dram_traffic("bwd_kernel<128>", name + "_backward", source_digest("bwd.cu", "ptx.cuh")),
                     "traffic_kernel": "bwd_kernel<128>",
                     "algorithmic_flops": flops},
        "gpu_launches": len(ts),
    }


def run_decode(steps, warmup, flush, peaks):
    import torch
    import exact_tiled_attention_15_gb300 as eta
    from exact_tiled_attention_15_gb300 import accounting as acc, workloads
    name = "gqa_decode"
    cfg = workloads.WORKLOADS[name]
    B, Hq, Hkv, D = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"]
    w = workloads.make_decode(B, Hq, Hkv, D, cfg["Lmin"], cfg["Lmax"], seed=0, poison_tail=False)
    dev = torch.device("cuda")
    q, kc, vc, sl = (w[n].to(dev) for n in ("q", "kcache", "vcache", "seqlens"))
    ws = torch.empty(eta.decode_workspace_bytes(B, Hq, Hkv, cfg["Lmax"], D), dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, device=dev, dtype=torch.float32)
    fn = lambda: eta.decode(q, kc, vc, sl, workspace=ws, out=o, lse_out=lse)  # noqa: E731
    ts = time_steps(fn, steps, warmup, flush, leg=name)
    if eta.get_error() != 0:
        raise RuntimeError("decode: device-side error")
    seqlens = w["seqlens"].tolist()
    nbytes = acc.decode_bytes(seqlens, B, Hq, Hkv, D)
    ms = statistics.mean(ts)
    gbs = nbytes / (ms * 1e-3) / 1e9
    digest = source_digest("decode.cu", "ptx.cuh")
    return {
        "metric": "KV-read GB/s (bf16 GQA decode)", "unit": "GB/s", "value": gbs,
        "ms_per_step": ms, **timing_stats(ts), "steps": len(ts),
        "config": {"workload": name, "B": B, "Hq": Hq, "Hkv": Hkv, "D": D, "Lmin": cfg["Lmin"],
                   "Lmax": cfg["Lmax"], "sum_seqlens": int(sum(seqlens))},
        "roofline": {"bound": "hbm", "kernel": "decode_split_kernel+decode_combine_kernel", "achieved": gbs,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                     "peak_source": peaks["source"] + " HBM copy",
                     "traffic": dram_traffic("decode_split_kernel", name, digest),
                     "algorithmic_bytes": nbytes},
        "gpu_launches": 2 * len(ts),
    }


def run_decode_paged(steps, warmup, flush, peaks):
    import torch
    import exact_tiled_attention_15_gb300 as eta
    from exact_tiled_attention_15_gb300 import accounting as acc, workloads
    name = "gqa_decode_paged"
    cfg = workloads.WORKLOADS[name]
    B, Hq, Hkv, D, ps = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["page_size"]
    w = workloads.make_paged_decode(B, Hq, Hkv, D, cfg["Lmin"], cfg["Lmax"], ps, seed=0, poison=False)
    dev = torch.device("cuda")
    t = {n: w[n].to(dev) for n in ("q", "k_pages", "v_pages", "block_table", "seqlens")}
    del w["kcache"], w["vcache"]
    ws = torch.empty(eta.decode_workspace_bytes(B, Hq, Hkv, t["block_table"].shape[1] * ps, D), dtype=torch.uint8,
                     device=dev)
    o = torch.empty_like(t["q"])
    lse = torch.empty(B, Hq, device=dev, dtype=torch.float32)
    fn = lambda: eta.decode_paged(t["q"], t["k_pages"], t["v_pages"], t["block_table"], t["seqlens"],  # noqa: E731
                                  workspace=ws, out=o, lse_out=lse)
    ts = time_steps(fn, steps, warmup, flush, leg=name)
    if eta.get_error() != 0:
        raise RuntimeError("paged decode: device-side error")
    seqlens = w["seqlens"].tolist()
    nbytes = acc.decode_bytes(seqlens, B, Hq, Hkv, D) + 4 * sum(-(-x // ps) for x in seqlens)
    ms = statistics.mean(ts)
    gbs = nbytes / (ms * 1e-3) / 1e9
    digest = source_digest("decode.cu", "ptx.cuh")
    return {
        "metric": "KV-read GB/s (bf16 GQA decode, paged KV cache)", "unit": "GB/s", "value": gbs,
        "ms_per_step": ms, **timing_stats(ts), "steps": len(ts),
        "config": {"workload": name, "B": B, "Hq": Hq, "Hkv": Hkv, "D": D, "Lmin": cfg["Lmin"],
                   "Lmax": cfg["Lmax"], "page_size": ps, "sum_seqlens": int(sum(seqlens))},
        "roofline": {"bound": "hbm", "kernel": "decode_split_kernel<128,paged>+decode_combine_kernel",
                     "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                     "peak_source": peaks["source"] + " HBM copy",
                     "traffic": dram_traffic("decode_split_kernel<128,paged>", name, digest),
                     "algorithmic_bytes": nbytes},
        "gpu_launches": 2 * len(ts),
    }


def run_decode_multi(steps, warmup, flush, peaks, T=4):
    import torch
    import exact_tiled_attention_15_gb300 as eta
    from exact_tiled_attention_15_gb300 import accounting as acc, workloads
    name = "gqa_decode"
    cfg = workloads.WORKLOADS[name]
    B, Hq, Hkv, D = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"]
    w = workloads.make_decode(B, Hq, Hkv, D, cfg["Lmin"], cfg["Lmax"], seed=0, poison_tail=False, T=T)
    dev = torch.device("cuda")
    q, kc, vc, sl = (w[n].to(dev) for n in ("q", "kcache", "vcache", "seqlens"))
    ws = torch.empty(int(eta.lib().attn_decode_multi_workspace_bytes(B, Hq, Hkv, T, cfg["Lmax"], D)),
                     dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, T, device=dev, dtype=torch.float32)
    fn = lambda: eta.decode_multi(q, kc, vc, sl, causal=True, workspace=ws, out=o, lse_out=lse)  # noqa: E731
    ts = time_steps(fn, steps, warmup, flush, leg=name + f"_T{T}")
    if eta.get_error() != 0:
        raise RuntimeError("multi-token decode: device-side error")
    seqlens = w["seqlens"].tolist()
    nbytes = acc.decode_bytes(seqlens, B, Hq * T, Hkv, D)
    ms = statistics.mean(ts)
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {
        "metric": f"KV-read GB/s (bf16 GQA decode, {T} causal query tokens per sequence)", "unit": "GB/s",
        "value": gbs, "ms_per_step": ms, **timing_stats(ts), "steps": len(ts),
        "config": {"workload": name + f"_T{T}", "B": B, "Hq": Hq, "Hkv": Hkv, "T": T, "D": D, "Lmin": cfg["Lmin"],
                   "Lmax": cfg["Lmax"], "sum_seqlens": int(sum(seqlens))},
        "roofline": {"bound": "hbm", "kernel": "decode_split_kernel+decode_combine_kernel (T query tokens)",
                     "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                     "peak_source": peaks["source"] + " HBM copy",
                     "traffic": dram_traffic("decode_split_kernel", name + f"_T{T}", source_digest("decode.cu", "ptx.cuh")),
                     "algorithmic_bytes": nbytes},
        "gpu_launches": 2 * len(ts),
    }


def run_quant(steps, warmup, flush, peaks):
    """Rotate + quantise Q, K (with signs) and V (without) of the FP8 workload."""
    import numpy as np
    import torch
    import exact_tiled_attention_15_gb300 as eta
    from exact_tiled_attention_15_gb300 import workloads
    cfg = workloads.WORKLOADS["fp8_prefill"]
    B, H, S, D = cfg["B"], cfg["Hq"], cfg["S"], cfg["D"]
    w = workloads.make_workload("fp8_prefill", seed=0)  # bf16 draws with 0.5 % outliers x50, and the signs
    dev = torch.device("cuda")
    xs = [w[n].to(dev) for n in ("q", "k", "v")]
    signs = torch.from_numpy(w["signs"].astype(np.float32)).to(dev)
    outs = [(torch.empty(B, H, S, D, dtype=torch.uint8, device=dev),
             torch.empty(B, H, -(-S // 128), 1, dtype=torch.float32, device=dev)) for _ in range(3)]

    def fn():  # Q and K rotated with the same signs, V not: one launch
        eta.rotate_quantize_fp8_many(xs, signs, rotate=(True, True, False), outs=outs)

    ts = time_steps(fn, steps, warmup, flush, leg="fp8_rotate_quantize")
    if eta.get_error() != 0:
        raise RuntimeError("rotate+quantise: device-side error")
    nbytes = 3 * (B * H * S * D * 3 + B * H * (-(-S // 128)) * 4)  # bf16 read + code write + scales
    ms = statistics.mean(ts)
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {
        "metric": "GB/s (Hadamard rotate + per-tile e4m3 quantise of Q, K, V)", "unit": "GB/s", "value": gbs,
        "ms_per_step": ms, **timing_stats(ts), "steps": len(ts),
        "config": {"workload": "fp8_prefill inputs", "B": B, "H": H, "S": S, "D": D, "tensors": 3},
        "roofline": {"bound": "hbm", "kernel": "rotate_quantize_kernel", "achieved": gbs, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"], "peak_source": peaks["source"] + " HBM copy",
                     # per step (one launch over Q, K, V), like algorithmic_bytes
                     "traffic": dram_traffic("rotate_quantize_kernel", "fp8_rotate_quantize",
                                             source_digest("quant.cu", "ptx.cuh")),
                     "algorithmic_bytes": nbytes},
        "gpu_launches": len(ts),
    }


def run_fp8(steps, warmup, flush, peaks):
    import torch
    import exact_tiled_attention_15_gb300 as eta
    from exact_tiled_attention_15_gb300 import accounting as acc, workloads
    name = "fp8_prefill"
    cfg = workloads.WORKLOADS[name]
    B, Hq, Hkv, S, D, causal = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["S"], cfg["D"], cfg["causal"]
    w = workloads.make_workload(name, seed=0)
    dev = torch.device("cuda")
    # the e4m3 inputs: Q and K rotated by the draw's signs, V not, by the library's quantise kernel
    signs = torch.from_numpy(w["signs"].astype("float32")).to(dev)
    (q8, qs), (k8, ks), (v8, vs) = eta.rotate_quantize_fp8_many([w[n].to(dev) for n in ("q", "k", "v")], signs,
                                                                rotate=(True, True, False))
    if eta.get_error() != 0:
        raise RuntimeError("fp8 inputs: device-side error")
    t = dict(q8=q8, k8=k8, v8=v8, q_scale=qs, k_scale=ks, v_scale=vs)
    o = torch.empty(B, Hq, S, D, device=dev, dtype=torch.bfloat16)
    lse = torch.empty(B, Hq, S, device=dev, dtype=torch.float32)
    fn = lambda: eta.fwd_fp8(t["q8"], t["k8"], t["v8"], t["q_scale"], t["k_scale"], t["v_scale"],  # noqa: E731
                             causal=causal, out=o, lse_out=lse)
    ts = time_steps(fn, steps, warmup, flush, leg=name)
    if eta.get_error() != 0:
        raise RuntimeError("fp8: device-side error")
    flops = acc.prefill_flops(B, Hq, S, S, D, causal)
    ms = statistics.mean(ts)
    ach = flops / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    digest = source_digest("fwd_kernel.cuh", "fwd_fp8.cu", "ptx.cuh")
    return {
        "metric": "attention TFLOP/s (FP8 e4m3 prefill)", "unit": "TFLOP/s", "value": ach,
        "ms_per_step": ms, **timing_stats(ts), "steps": len(ts),
        "config": {"workload": name, "B": B, "Hq": Hq, "Hkv": Hkv, "Sq": S, "Sk": S, "D": D, "causal": causal},
        "roofline": {"bound": "tensor", "kernel": "fwd_kernel<Fp8,128>", "achieved": ach, "peak": peak,
                     "unit": "TFLOP/s", "frac": ach / peak,
                     "peak_source": peaks["source"] + " bf16 burst x 2 (nominal FP8/BF16 ratio)",
                     "traffic": dram_traffic("fwd_kernel<Fp8,128>", name, digest),
                     "algorithmic_bytes": acc.prefill_bytes(B, Hq, Hkv, S, S, D, elem_bytes=1)
                     + acc.fp8_scale_bytes(B, Hq, Hkv, S, S, D)},
        "gpu_launches": len(ts),
    }


# ---------------------------------------------------------------- CPU oracle
_INPUT_CACHE = {}
_GPU_OUT = {}  # workload -> (O, LSE) of its last timed GPU step, on the host


def sample_parity(name, heads, O, L):
    """The timed run's GPU output against the oracle's on the sampled (b, h)
    heads: max |dO| element by element, graded against 1e-2 plus half a bf16
    ulp of the oracle's O (the output's own rounding), and max |dLSE| against
    1e-3; None if the workload's output was not kept."""
    import numpy as np
    if name not in _GPU_OUT:
        return None
    o, lse = _GPU_OUT[name]
    go = np.stack([o[b, h].double().numpy() for b, h in heads])
    gl = np.stack([lse[b, h].double().numpy() for b, h in heads])
    d = np.abs(go - O)
    ax = np.abs(O)
    half_ulp = np.where(ax > 0, np.exp2(np.floor(np.log2(np.where(ax > 0, ax, 1.0))) - 8), 0.0)
    fin = np.isfinite(L)
    same_inf = bool((np.isneginf(gl) == np.isneginf(L)).all())
    dl = float(np.abs(gl[fin] - L[fin]).max()) if fin.any() else 0.0
    return {"heads": len(heads), "elements": int(d.size), "max_abs_dO": float(d.max()),
            "elements_over_1e-2": int((d > 1e-2).sum()), "max_abs_dLSE": dl,
            "within_bound": bool((d <= 1e-2 + half_ulp).all() and dl <= 1e-3 and same_inf)}


def oracle_head_sample(name, budget_s=10.0, max_heads=None):
    """The fp64 oracle over whole (b, h) heads of the workload, one head after
    another (BLAS threads on the host cores), until budget_s has elapsed;
    returns (TFLOP/s, heads, seconds, cores, flops)."""
    import numpy as np
    import oracle
    from exact_tiled_attention_15_gb300 import accounting as acc, workloads
    cfg = workloads.WORKLOADS[name]
    if name not in _INPUT_CACHE:
        _INPUT_CACHE[name] = workloads.make_workload(name, seed=0)
    w = _INPUT_CACHE[name]
    S, D, causal = cfg["S"], cfg["D"], cfg["causal"]
    g = cfg["Hq"] // cfg["Hkv"]
    heads, t_total = 0, 0.0
    order = [(b, h) for b in range(cfg["B"]) for h in range(cfg["Hq"])]
    for b, h in order:
        qh = w["q"][b:b + 1, h:h + 1].double().numpy()
        kh = w["k"][b:b + 1, h // g:h // g + 1].double().numpy()
        vh = w["v"][b:b + 1, h // g:h // g + 1].double().numpy()
        t0 = time.perf_counter()
        oracle.attention(qh, kh, vh, causal=causal, scale=1.0 / math.sqrt(D))
        t_total += time.perf_counter() - t0
        heads += 1
        if t_total >= budget_s or (max_heads and heads >= max_heads):
            break
    flops = acc.prefill_flops(1, heads, S, S, D, causal)
    cores = len(os.sched_getaffinity(0))
    return flops / t_total / 1e12, heads, t_total, cores, flops


def oracle_pool_sample(name, budget_s=10.0):
    """The fp64 oracle over whole heads of the workload on a process pool of
    one single-threaded worker per host core (heads are independent problems):
    after one untimed round (one head per worker, which also starts them),
    rounds of one head per worker until budget_s has elapsed.  Returns
    (TFLOP/s, heads, seconds, workers, flops, last round's heads, their O, LSE)."""
    from exact_tiled_attention_15_gb300 import accounting as acc, workloads
    from oracle.pool import HeadPool
    cfg = workloads.WORKLOADS[name]
    if name not in _INPUT_CACHE:
        _INPUT_CACHE[name] = workloads.make_workload(name, seed=0)
    w = _INPUT_CACHE[name]
    S, D, causal = cfg["S"], cfg["D"], cfg["causal"]
    order = [(b, h) for b in range(cfg["B"]) for h in range(cfg["Hq"])]
    with HeadPool(w["q"].float().numpy(), w["k"].float().numpy(), w["v"].float().numpy()) as pool:
        n = pool.workers
        pool.run(order[:n], causal, 1.0 / math.sqrt(D))
        done, t, r = 0, 0.0, 1
        batch, O, L = [], None, None
        while t < budget_s:
            batch = [order[(r * n + i) % len(order)] for i in range(n)]
            t0 = time.perf_counter()
            O, L = pool.run(batch, causal, 1.0 / math.sqrt(D))
            t += time.perf_counter() - t0
            done += n
            r += 1
    flops = acc.prefill_flops(1, done, S, S, D, causal)
    return flops / t / 1e12, done, t, n, flops, batch, O, L


def headline_config(ws):
    """The `config` object of the headline line (both arms)."""
    from exact_tiled_attention_15_gb300 import workloads
    cfg = workloads.WORKLOADS[HEADLINE]
    return {"workload": HEADLINE, "B": cfg["B"], "Hq": cfg["Hq"], "Hkv": cfg["Hkv"], "Sq": cfg["S"], "Sk": cfg["S"],
            "D": cfg["D"], "causal": cfg["causal"],
            "l2": "flushed between steps outside the timed events (256 MB write, then 256 MB read of another "
                  "buffer: clean L2 without the inputs); inputs 402 MB also exceed the 129 MB L2",
            "parallelism": f"replicas x{ws}"}


def reference_arm(args, ws, rank):
    """--impl reference: the CPU fp64 oracle as it stands, one head of the
    headline workload per step, on this machine's host cores."""
    if rank != 0:
        return
    for _ in range(args.warmup):
        oracle_head_sample(HEADLINE, budget_s=0.0, max_heads=1)
    t0 = time.perf_counter()
    tot_flops, tot_t, heads, cores = 0.0, 0.0, 0, 1
    for _ in range(args.steps):
        _, h, t, cores, f = oracle_head_sample(HEADLINE, budget_s=0.0, max_heads=1)
        tot_flops += f
        tot_t += t
        heads += h
    wall = time.perf_counter() - t0
    value = tot_flops / tot_t / 1e12
    sample = f"{heads} step(s) of one full causal head (b=0, h=0; 4096 x 4096 scores, D=128) of the headline workload"
    line = {
        "impl": "reference", "metric": HEADLINE_METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_t / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": headline_config(ws),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": wall,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- main
def main():
    args = parse_args()
    ws, rank, local = dist_setup(args)
    if args.impl == "reference":
        reference_arm(args, ws, rank)
        return
    import torch
    peaks = load_peaks()
    flush = L2Flush()
    if args.only:
        if args.only == "gqa_decode":
            res = run_decode(args.steps, args.warmup, flush, peaks)
        elif args.only == "chunked_prefill":
            res = run_chunked_prefill(args.steps, args.warmup, flush, peaks)
        elif args.only == "train_prefill_mha_backward":
            res = run_backward(args.steps, args.warmup, flush, peaks)
        elif args.only == "gqa_decode_paged":
            res = run_decode_paged(args.steps, args.warmup, flush, peaks)
        elif args.only == "fp8_rotate_quantize":
            res = run_quant(args.steps, args.warmup, flush, peaks)
        elif args.only == "gqa_decode_T4":
            res = run_decode_multi(args.steps, args.warmup, flush, peaks, T=4)
        elif args.only == "fp8_prefill":
            res = run_fp8(args.steps, args.warmup, flush, peaks)
        else:
            res = run_prefill(args.only, args.steps, args.warmup, flush, peaks,
                              e2e_steps=args.e2e_steps if args.only == HEADLINE else 0)
        if rank == 0:
            add_spec(res.get("roofline"))
            print(json.dumps(dict(res, only=args.only)), flush=True)
        return
    clocks = ClockSampler(local)
    clocks.start()
    nvml = NvmlClockSampler(local)
    nvml.start()
    time.sleep(0.3)
    barrier(ws)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    head = run_prefill(HEADLINE, args.steps, args.warmup, flush, peaks)
    torch.cuda.synchronize()
    barrier(ws)
    region_s = time.perf_counter() - t0
    step_ms = max_over_ranks(head["ms_per_step"], ws)
    extras = {}
    if not args.no_extras:
        extras["long_gqa_prefill"] = run_prefill("long_gqa_prefill", max(5, args.steps // 4), args.warmup, flush, peaks)
        extras["chunked_prefill"] = run_chunked_prefill(args.steps, args.warmup, flush, peaks)
        extras["train_prefill_mha_backward"] = run_backward(max(5, args.steps // 4), args.warmup, flush, peaks)
        extras["gqa_decode"] = run_decode(args.steps, args.warmup, flush, peaks)
        extras["gqa_decode_paged"] = run_decode_paged(args.steps, args.warmup, flush, peaks)
        extras["gqa_decode_T4"] = run_decode_multi(args.steps, args.warmup, flush, peaks, T=4)
        extras["fp8_rotate_quantize"] = run_quant(args.steps, args.warmup, flush, peaks)
        try:
            extras["fp8_prefill"] = run_fp8(args.steps, args.warmup, flush, peaks)
        except Exception as e:  # reported, not hidden
            extras["fp8_prefill"] = {"error": str(e).splitlines()[0]}
    e2e = None
    if args.e2e_steps > 0:
        e2e = run_prefill(HEADLINE, 1, 1, flush, peaks, e2e_steps=args.e2e_steps, leg=None)["e2e"]
    nvml.stop()
    clk = clocks.stop()
    if rank != 0:
        return
    add_spec(head["roofline"])
    for leg in extras.values():
        if isinstance(leg, dict) and "roofline" in leg:
            add_spec(leg["roofline"])
    # clock samples binned by each leg's timed steps (NVML, ~1 ms apart)
    leg_clk = {name: nvml.window(*win) for name, win in LEG_WINDOWS.items()} if nvml.ok else {}
    head_clk = leg_clk.get(HEADLINE, {})
    value = whole_job_tflops(head["flops_per_step"], ws, step_ms)
    reasons = sorted(set(clk["reasons"]) | {r for c in leg_clk.values() for r in c["reasons"]})
    line = {
        "metric": HEADLINE_METRIC,
        "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_ms, "ms_median": head["ms_median"], "ms_p95": head["ms_p95"],
        "ms_ci95": head["ms_ci95"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": headline_config(ws),
        "roofline": head["roofline"],
        "e2e": None if e2e is None else {
            "value": e2e["value"] * ws, "unit": "TFLOP/s", "h2d_bytes_per_step": e2e["h2d_bytes_per_step"],
            "d2h_bytes_per_step": e2e["d2h_bytes_per_step"], "ms_per_step": e2e["ms_per_step"],
            "api": e2e["api"], "equals_device_output": e2e.get("equals_device_output")},
        "gpu_launches": head["gpu_launches"],
        "clocks": {"sm_mhz": head_clk.get("sm_mhz") or clk["sm_mhz"],
                   "sm_max_mhz": getattr(nvml, "sm_max", None) or clk["sm_max_mhz"], "reasons": reasons,
                   "samples": head_clk.get("samples", clk["samples"]),
                   "how": ("NVML every ~1 ms inside the headline's timed steps" if head_clk.get("samples")
                           else "nvidia-smi every 200 ms over the run"),
                   "smi_sm_mhz_median": clk["sm_mhz"], "smi_samples": clk["samples"]},
        "workloads": extras,
        "timed_region_s": region_s,
    }
    if not args.no_cpu_baseline and ws == 1:
        v, heads, t, cores, _, last, Oref, Lref = oracle_pool_sample(HEADLINE, budget_s=10.0)
        line["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "sample": f"{heads} full causal heads of the headline workload in {t:.1f} s: "
                                          f"the fp64 NumPy oracle on {cores} single-threaded worker processes, "
                                          f"one head each at a time",
                                "parity": sample_parity(HEADLINE, last, Oref, Lref)}
    # last: one short entry per leg, so every figure survives a cut of the line's head
    legs = {HEADLINE: head, **extras}
    line["legs_fields"] = ["value", "unit", "roofline frac (measured peak)", "ms per step", "median SM MHz"]
    line["legs"] = {}
    for name, r in legs.items():
        if not isinstance(r, dict) or "value" not in r:
            line["legs"][name] = r
            continue
        c = leg_clk.get(name, {})
        line["legs"][name] = [round(r["value"], 1), r["unit"], round(r["roofline"]["frac"], 3),
                              round(r["ms_per_step"], 4), c.get("sm_mhz")]
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
