"""GPU parity of the fused Hadamard-rotate + per-tile e4m3 quantise kernel
against the fp64 oracle.

Codes are bytes, so they must match exactly -- except where the exact value
y / scale lies so close to an e4m3 rounding boundary that the kernel's fp32
transform (a different summation order than the oracle's) may land on either
side; there both neighbouring codes are valid, and the test counts them.

The kernel forms z = x H diag(s) on the tensor core: the 128 products are
exact (bf16 times +-1) and are summed in fp32 in an order and with a rounding
that the hardware does not document.  The band assumes each product enters
the sum with at most one truncation (relative 2^-23) of a partial sum no
larger than sum |x|: |z - z_exact| <= 128 * 2^-23 * sum |x|.  Measured through
a copy of the kernel that wrote z out: at most 2.1 * 2^-24 * sum |x| on rows
like the workload's and 18.7 on adversarial rows (one entry 2^24 times the
other 127), against the 256 assumed here."""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_15_gb300 import workloads

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def signs_for(seed, D=128):
    return np.random.default_rng(seed).integers(0, 2, D).astype(np.float64) * 2 - 1


def check(x_bf16, signs, codes_gpu, scales_gpu, what):
    x = x_bf16.double().numpy()
    codes, scales, y = oracle.rotate_quantize(x, signs)
    # the transform's error bound (module docstring); then y = z / sqrt(D), 1 / scale
    # and y * (1 / scale) are each rounded once (3 half-ulps, rounded up to 4)
    # (a 64-wide head is summed over 128 products too, half of them zero)
    eps = 256 * 2.0 ** -24 * np.abs(x).sum(-1, keepdims=True) / np.sqrt(x.shape[-1]) + 2.0 ** -22 * np.abs(y)
    S = x.shape[2]
    pad = -S % 128
    eps_tile = np.pad(eps.max(-1), ((0, 0), (0, 0), (0, pad))).reshape(*x.shape[:2], -1, 128).max(-1)[..., None]
    sg = scales_gpu.double().numpy()
    # scale = max |y| / 448: off by at most the tile's largest eps / 448, plus its own rounding
    assert (np.abs(sg - scales) <= eps_tile / 448 + 2.0 ** -22 * scales).all(), what
    cg = codes_gpu.numpy()
    exact = cg == codes
    if not exact.all():
        sc = np.repeat(sg, 128, axis=2)[:, :, :S]
        # rounding is monotone: every code from that of (y - eps) to that of (y + eps)
        # is a correct rounding of a value inside the band
        lo = oracle.e4m3_decode(oracle.e4m3_encode((y - eps) / sc))
        hi = oracle.e4m3_decode(oracle.e4m3_encode((y + eps) / sc))
        v = oracle.e4m3_decode(cg)
        ok = exact | ((v >= lo) & (v <= hi))
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


@pytest.mark.parametrize("S", [300, 1000])
@pytest.mark.parametrize("rotate", [True, False])
def test_rotate_quantize_head_dim_64(S, rotate):
    """D = 64: the kernel reads 128-column tiles whose upper half arrives as
    zeros and rotates by H_64 diag(s) / 8, the leading block of its matrix;
    only the 64 real columns of codes are stored."""
    import exact_tiled_attention_15_gb300 as eta
    rng = np.random.default_rng(S + 64)
    x = rng.standard_normal((2, 3, S, 64)).astype(np.float32)
    x[rng.random(x.shape) < 0.005] *= 50.0
    xb = workloads.to_bf16(x)
    signs = signs_for(S, 64) if rotate else None
    sg = torch.from_numpy(signs.astype(np.float32)).to(DEV) if rotate else None
    codes, scales = eta.rotate_quantize_fp8(xb.to(DEV), sg)
    assert eta.get_error() == 0
    assert codes.shape == (2, 3, S, 64) and scales.shape == (2, 3, -(-S // 128), 1)
    check(xb, signs, codes.cpu(), scales.cpu(), f"D=64 S={S} rotate={rotate}")
    many = eta.rotate_quantize_fp8_many([xb.to(DEV), xb.to(DEV)], sg if rotate else None, rotate=[rotate, False])
    assert eta.get_error() == 0
    assert torch.equal(many[0][0], codes) and torch.equal(many[0][1], scales)
    check(xb, None, many[1][0].cpu(), many[1][1].cpu(), f"D=64 S={S} many, identity")


def test_wide_dynamic_range_rows():
    """Rows whose entries span many binades (one entry per row 2^24 times the
    rest, and heavy-tailed magnitudes): the tensor core's alignment of small
    terms to large partial sums is where its accumulation loses most."""
    import exact_tiled_attention_15_gb300 as eta
    rng = np.random.default_rng(11)
    x = (rng.choice([-1.0, 1.0], (1, 2, 512, 128)) * 2.0 ** -12 * (1 + rng.random((1, 2, 512, 128))))
    idx = rng.integers(0, 128, (1, 2, 512))
    np.put_along_axis(x, idx[..., None], 2.0 ** 12 * (1 + rng.random((1, 2, 512, 1))), -1)
    x[:, 1] = rng.standard_normal((1, 512, 128)) * 2.0 ** rng.uniform(-12, 0, (1, 512, 128))
    xb = workloads.to_bf16(x.astype(np.float32))
    signs = signs_for(11)
    codes, scales = eta.rotate_quantize_fp8(xb.to(DEV), torch.from_numpy(signs.astype(np.float32)).to(DEV))
    assert eta.get_error() == 0
    check(xb, signs, codes.cpu(), scales.cpu(), "wide dynamic range")


def test_many_tensors_one_launch_matches_single_calls():
    """attn_rotate_quantize_fp8_many: Q and K rotated with the same signs, V not,
    of different head counts and ragged lengths, in one launch -- byte for byte
    the single-tensor results, and checked against the oracle."""
    import exact_tiled_attention_15_gb300 as eta
    rng = np.random.default_rng(5)
    shapes = [(2, 4, 300, 128), (2, 2, 1000, 128), (2, 2, 1000, 128), (1, 1, 1, 128)]
    xs = []
    for sh in shapes:
        x = rng.standard_normal(sh).astype(np.float32)
        x[rng.random(x.shape) < 0.005] *= 50.0
        xs.append(workloads.to_bf16(x))
    signs = signs_for(5)
    sg = torch.from_numpy(signs.astype(np.float32)).to(DEV)
    rotate = [True, True, False, True]
    many = eta.rotate_quantize_fp8_many([x.to(DEV) for x in xs], sg, rotate=rotate)
    assert eta.get_error() == 0
    for i, (x, r, (c, sc)) in enumerate(zip(xs, rotate, many)):
        c1, s1 = eta.rotate_quantize_fp8(x.to(DEV), sg if r else None)
        assert torch.equal(c, c1) and torch.equal(sc, s1), f"tensor {i}"
        check(x, signs if r else None, c.cpu(), sc.cpu(), f"many[{i}]")


def test_all_zero_tile_and_constant_rows():
    import exact_tiled_attention_15_gb300 as eta
    x = torch.zeros(1, 1, 256, 128, dtype=torch.bfloat16)
    x[0, 0, 128:] = 3.0  # second tile: constant rows (the transform puts all mass in column 0)
    signs = signs_for(7)
    codes, scales = eta.rotate_quantize_fp8(x.to(DEV), torch.from_numpy(signs.astype(np.float32)).to(DEV))
    assert scales[0, 0, 0, 0].item() == 1.0 and (codes[0, 0, :128] == 0).all()
    check(x, signs, codes.cpu(), scales.cpu(), "zero / constant tiles")


def test_full_size_q_and_fp8_attention_end_to_end():
    """The FP8 workload's Q, K (rotated with the same signs) and V (not), each
    B=2, H=16, S=8192, quantised on the GPU and checked code by code (every
    code of all three tensors); then they feed the FP8 attention, checked
    against the oracle on the dequantised codes."""
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
    for name, x, sg_, (c, sc) in zip("QKV", xs, (signs, signs, None), out):
        n_edge = check(x, sg_, c.cpu(), sc.cpu(), f"full-size {name}")
        print(f"full-size {name}: {n_edge} of {x.numel()} codes on a rounding boundary")
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
