"""GPU parity of the fused Hadamard-rotate + per-tile e4m3 quantise kernel
against the fp64 oracle.

Codes are bytes, so they must match exactly -- except where the exact value
y / scale lies so close to an e4m3 rounding boundary that the kernel's fp32
transform (a different summation order than the oracle's) may land on either
side; there both neighbouring codes are valid, and the test counts them."""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_15_gb300 import workloads

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def signs_for(seed):
    return np.random.default_rng(seed).integers(0, 2, 128).astype(np.float64) * 2 - 1


def check(x_bf16, signs, codes_gpu, scales_gpu, what):
    x = x_bf16.double().numpy()
    codes, scales, y = oracle.rotate_quantize(x, signs)
    sg = scales_gpu.double().numpy()
    np.testing.assert_allclose(sg, scales, rtol=1e-5, err_msg=what)
    cg = codes_gpu.numpy()
    exact = cg == codes
    if not exact.all():
        # fp32 error bound of the transform: a sum of 128 terms over 7 levels
        eps = 8 * 2.0 ** -24 * np.abs(x).sum(-1, keepdims=True) / np.sqrt(128) + 2.0 ** -23 * np.abs(y)
        sc = np.repeat(sg, 128, axis=2)[:, :, :x.shape[2]]
        lo = oracle.e4m3_encode((y - eps) / sc)
        hi = oracle.e4m3_encode((y + eps) / sc)
        ok = exact | (cg == lo) | (cg == hi)
        assert ok.all(), f"{what}: {(~ok).sum()} codes outside the rounding tolerance"
    return int((~exact).sum())


@pytest.mark.parametrize("S", [1, 128, 300, 1000])
@pytest.mark.parametrize("rotate", [True, False])
def test_rotate_quantize_shapes(S, rotate):
    import exact_tiled_attention_15_gb300 as eta
    rng = np.random.default_rng(S)
    x = rng.standard_normal((1, 3, S, 128)).astype(np.float32)
    x[rng.random(x.shape) < 0.005] *= 50.0
    xb = workloads.to_bf16(x)
    signs = signs_for(S) if rotate else None
    sg = torch.from_numpy(signs.astype(np.float32)).to(DEV) if rotate else None
    codes, scales = eta.rotate_quantize_fp8(xb.to(DEV), sg)
    assert eta.get_error() == 0
    check(xb, signs, codes.cpu(), scales.cpu(), f"S={S} rotate={rotate}")


def test_all_zero_tile_and_constant_rows():
    import exact_tiled_attention_15_gb300 as eta
    x = torch.zeros(1, 1, 256, 128, dtype=torch.bfloat16)
    x[0, 0, 128:] = 3.0  # second tile: constant rows (the transform puts all mass in column 0)
    signs = signs_for(7)
    codes, scales = eta.rotate_quantize_fp8(x.to(DEV), torch.from_numpy(signs.astype(np.float32)).to(DEV))
    assert scales[0, 0, 0, 0].item() == 1.0 and (codes[0, 0, :128] == 0).all()
    check(x, signs, codes.cpu(), scales.cpu(), "zero / constant tiles")


def test_full_size_q_and_fp8_attention_end_to_end():
    """The FP8 workload's Q (B=2, H=16, S=8192) rotated and quantised on the
    GPU, checked code by code; then Q, K (rotated) and V (not) feed the FP8
    attention, checked against the oracle on the dequantised codes."""
    import exact_tiled_attention_15_gb300 as eta
    rng = np.random.default_rng(0)
    B, H, S, D = 2, 16, 8192, 128
    xs = []
    for _ in range(3):
        x = rng.standard_normal((B, H, S, D)).astype(np.float32)
        x[rng.random(x.shape) < 0.005] *= 50.0
        xs.append(workloads.to_bf16(x))
    signs = signs_for(1)
    sg = torch.from_numpy(signs.astype(np.float32)).to(DEV)
    out = [eta.rotate_quantize_fp8(xs[0].to(DEV), sg), eta.rotate_quantize_fp8(xs[1].to(DEV), sg),
           eta.rotate_quantize_fp8(xs[2].to(DEV), None)]
    assert eta.get_error() == 0
    n_edge = check(xs[0], signs, out[0][0].cpu(), out[0][1].cpu(), "full-size Q")
    print(f"full-size Q: {n_edge} of {xs[0].numel()} codes on a rounding boundary")
    o, lse = eta.fwd_fp8(out[0][0], out[1][0], out[2][0], out[0][1], out[1][1], out[2][1])
    assert eta.get_error() == 0
    o = o.double().cpu().numpy()
    rows = np.array([0, 1, 777, 4096, 8191])
    for b, h in [(0, 0), (1, 11)]:
        deq = [oracle.dequantize_tiles(c[b:b + 1, h:h + 1].cpu().numpy(), s[b:b + 1, h:h + 1].cpu().numpy())
               for c, s in out]
        Or, _ = oracle.attention_rows(deq[0], deq[1], deq[2], 0, 0, rows, False, 1 / np.sqrt(D))
        rr = np.linalg.norm(o[b, h, rows] - Or) / np.linalg.norm(Or)
        assert rr <= 5e-2, rr
