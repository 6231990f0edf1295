"""Tolerances of the GPU-vs-oracle parity tests.

bf16 outputs: |O_gpu - O_ref| <= 1e-2 + half a bf16 ulp of O_ref, elementwise.
The 1e-2 is the stated bound for bf16 inputs with fp32 accumulation; the
half-ulp term is the rounding of the output itself to bf16 (8 significant
bits), which alone exceeds 1e-2 once |O| >= 4.  LSE (fp32): |dLSE| <= 1e-3.
FP8 outputs: ||O_gpu - O_ref||_F / ||O_ref||_F <= 5e-2 over the whole tensor.
"""
import numpy as np

O_ABS = 1e-2
LSE_ABS = 1e-3
FP8_REL_RMS = 5e-2


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, np.exp2(e - 8), 0.0)


def check_bf16(o_gpu, o_ref, lse_gpu=None, lse_ref=None, what=""):
    """Assert the bf16 bound; returns (max |dO|, max |dLSE|)."""
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    assert o_gpu.shape == o_ref.shape, (o_gpu.shape, o_ref.shape)
    assert np.isfinite(o_gpu).all(), f"{what}: non-finite output"
    err = np.abs(o_gpu - o_ref)
    bound = O_ABS + half_ulp_bf16(o_ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outputs beyond bound; "
                           f"max err {err.max():.3g} at {np.unravel_index(err.argmax(), err.shape)}")
    dl = 0.0
    if lse_ref is not None:
        lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
        lse_ref = np.asarray(lse_ref, dtype=np.float64)
        same_inf = np.isneginf(lse_gpu) == np.isneginf(lse_ref)
        assert same_inf.all(), f"{what}: -inf pattern of LSE differs"
        fin = np.isfinite(lse_ref)
        if fin.any():
            dl = float(np.abs(lse_gpu[fin] - lse_ref[fin]).max())
        assert dl <= LSE_ABS, f"{what}: LSE max err {dl:.3g}"
    return float(err.max()), dl


def rel_rms(o_gpu, o_ref) -> float:
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    return float(np.linalg.norm(o_gpu - o_ref) / np.linalg.norm(o_ref))
