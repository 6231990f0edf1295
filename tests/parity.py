"""Tolerances of the GPU-vs-oracle parity tests.

bf16 outputs: |O_gpu - O_ref| <= 1e-2 + half a bf16 ulp of O_ref, elementwise.
The 1e-2 is the stated bound for bf16 inputs with fp32 accumulation; the
half-ulp term is the rounding of the output itself to bf16 (8 significant
bits), which alone exceeds 1e-2 once |O| >= 4.  Every check reports the plain
max |O_gpu - O_ref| beside it, and how many elements lay above 1e-2 and so
needed the half-ulp term.  LSE (fp32): |dLSE| <= 1e-3.
FP8 outputs: ||O_gpu - O_ref||_F / ||O_ref||_F <= 5e-2 over the whole tensor.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

O_ABS = 1e-2
LSE_ABS = 1e-3
FP8_REL_RMS = 5e-2


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, np.exp2(e - 8), 0.0)


@dataclass
class Bf16Report:
    """What one or more bf16 checks saw."""
    max_abs: float = 0.0    # plain max |O_gpu - O_ref|
    max_lse: float = 0.0    # max |LSE_gpu - LSE_ref| over finite rows
    n_half_ulp: int = 0     # elements with |dO| > 1e-2 (inside 1e-2 + half ulp)
    n: int = 0              # elements compared

    def merge(self, other: "Bf16Report") -> "Bf16Report":
        return Bf16Report(max(self.max_abs, other.max_abs), max(self.max_lse, other.max_lse),
                          self.n_half_ulp + other.n_half_ulp, self.n + other.n)

    def __str__(self):
        return (f"max|dO| {self.max_abs:.4g} (plain), {self.n_half_ulp} of {self.n} elements above 1e-2 "
                f"within the half-ulp term, max|dLSE| {self.max_lse:.3g}")


def check_bf16(o_gpu, o_ref, lse_gpu=None, lse_ref=None, what="") -> Bf16Report:
    """Assert the bf16 bound; returns what was seen (plain max-abs error, the
    count of elements that needed the half-ulp term, max LSE error)."""
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    assert o_gpu.shape == o_ref.shape, (o_gpu.shape, o_ref.shape)
    assert np.isfinite(o_gpu).all(), f"{what}: non-finite output"
    err = np.abs(o_gpu - o_ref)
    bound = O_ABS + half_ulp_bf16(o_ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outputs beyond bound; "
                           f"max err {err.max():.3g} at {np.unravel_index(err.argmax(), err.shape)}")
    rep = Bf16Report(float(err.max()) if err.size else 0.0, 0.0, int((err > O_ABS).sum()), int(err.size))
    if lse_ref is not None:
        lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
        lse_ref = np.asarray(lse_ref, dtype=np.float64)
        same_inf = np.isneginf(lse_gpu) == np.isneginf(lse_ref)
        assert same_inf.all(), f"{what}: -inf pattern of LSE differs"
        fin = np.isfinite(lse_ref)
        if fin.any():
            rep.max_lse = float(np.abs(lse_gpu[fin] - lse_ref[fin]).max())
        assert rep.max_lse <= LSE_ABS, f"{what}: LSE max err {rep.max_lse:.3g}"
    return rep


def rel_rms(o_gpu, o_ref) -> float:
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    return float(np.linalg.norm(o_gpu - o_ref) / np.linalg.norm(o_ref))


def fp8_inputs(w):
    """The FP8 prefill inputs of a ``workloads.make_fp8_prefill`` draw, made by
    the oracle's rotate + quantise (Q and K rotated by the draw's signs, V
    not; one fp32 scale per 128 x 128 tile), as CPU tensors keyed q8, k8, v8,
    q_scale, k_scale, v_scale.  The GPU and the oracle then both consume these
    codes and scales, so neither side's inputs come from the other."""
    import torch

    import oracle
    out = {}
    for n, signs in (("q", w["signs"]), ("k", w["signs"]), ("v", None)):
        codes, scales, _ = oracle.rotate_quantize(w[n].double().numpy(), signs)
        out[n + "8"] = torch.from_numpy(codes)
        out[n + "_scale"] = torch.from_numpy(scales.astype(np.float32))
    return out
