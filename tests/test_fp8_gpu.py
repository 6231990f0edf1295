"""GPU parity of the FP8 e4m3 prefill kernel against the fp64 oracle on the
dequantised inputs (code x tile scale)."""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_15_gb300 import workloads
from parity import FP8_REL_RMS, LSE_ABS, fp8_inputs, rel_rms

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
NAMES = ("q8", "k8", "v8", "q_scale", "k_scale", "v_scale")


def deq(w, name, b=None, h=None):
    codes, scales = w[name + "8"], w[name + "_scale"]
    if b is not None:
        codes, scales = codes[b:b + 1, h:h + 1], scales[b:b + 1, h:h + 1]
    return oracle.dequantize_tiles(codes.numpy(), scales.numpy())


def gpu_fp8(w, causal):
    import exact_tiled_attention_15_gb300 as eta
    t = [w[n].to(DEV) for n in NAMES]
    o, lse = eta.fwd_fp8(*t, causal=causal)
    assert eta.get_error() == 0
    return o.double().cpu().numpy(), lse.cpu().numpy()


def check(o, lse, Or, Lr, what):
    assert np.isfinite(o).all(), what
    rr = rel_rms(o, Or)
    assert rr <= FP8_REL_RMS, f"{what}: relative RMS {rr:.4f}"
    fin = np.isfinite(Lr)
    assert (np.isneginf(lse) == np.isneginf(Lr)).all(), what
    dl = np.abs(lse[fin] - Lr[fin]).max() if fin.any() else 0.0
    assert dl <= LSE_ABS, f"{what}: LSE max err {dl:.3g}"
    return rr, dl


@pytest.mark.parametrize("S", [1, 128, 300, 1000])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_shapes(S, causal):
    w = fp8_inputs(workloads.make_fp8_prefill(1, 2, 2, S, S, 128, seed=S))
    o, lse = gpu_fp8(w, causal)
    Or, Lr = oracle.attention(deq(w, "q"), deq(w, "k"), deq(w, "v"), causal=causal)
    check(o, lse, Or, Lr, f"fp8 S={S} causal={causal}")


@pytest.mark.parametrize("Sq,Sk", [(100, 700), (700, 100)])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_gqa_unequal(Sq, Sk, causal):
    w = fp8_inputs(workloads.make_fp8_prefill(2, 4, 2, Sq, Sk, 128, seed=Sq))
    o, lse = gpu_fp8(w, causal)
    Or, Lr = oracle.attention(deq(w, "q"), deq(w, "k"), deq(w, "v"), causal=causal)
    check(o, lse, Or, Lr, f"fp8 {Sq}x{Sk} causal={causal}")


@pytest.mark.parametrize("Sq,Sk", [(300, 300), (100, 700), (700, 100)])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_head_dim_64(Sq, Sk, causal):
    """D = 64 on the D = 128 kernel: 128-column tiles whose upper half TMA
    reads as zeros (nothing added to Q K^T, O's upper half zero); only the
    64 real columns of O are written, at a row stride of 64."""
    w = fp8_inputs(workloads.make_fp8_prefill(2, 4, 2, Sq, Sk, 64, seed=Sq + Sk))
    assert w["q_scale"].shape == (2, 4, -(-Sq // 128), 1)
    o, lse = gpu_fp8(w, causal)
    assert o.shape == (2, 4, Sq, 64)
    Or, Lr = oracle.attention(deq(w, "q"), deq(w, "k"), deq(w, "v"), causal=causal)
    check(o, lse, Or, Lr, f"fp8 D=64 {Sq}x{Sk} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_many_key_tiles_gqa(causal):
    """17 key tiles (the last one ragged), query groups of 4: the three-stage
    K and V rings wrap several times with K slots handed back by the V
    release, and under the causal mask the two Q tiles of a CTA visit
    different numbers of key tiles."""
    w = fp8_inputs(workloads.make_fp8_prefill(1, 8, 2, 2100, 2100, 128, seed=21))
    o, lse = gpu_fp8(w, causal)
    Or, Lr = oracle.attention(deq(w, "q"), deq(w, "k"), deq(w, "v"), causal=causal)
    check(o, lse, Or, Lr, f"fp8 2100 GQA 8/2 causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_running_max_jump(causal):
    """As for bf16: later key tiles x60 make the running max jump past the
    exp2 range, so the accumulated O must be multiplied by an underflowed 0."""
    rng = np.random.default_rng(9)
    q = torch.from_numpy(rng.standard_normal((1, 2, 400, 128)).astype(np.float32))
    k = torch.from_numpy(rng.standard_normal((1, 2, 400, 128)).astype(np.float32))
    v = torch.from_numpy(rng.standard_normal((1, 2, 400, 128)).astype(np.float32))
    k[:, :, 128:] *= 60.0
    w = {}
    for n, x in (("q", q), ("k", k), ("v", v)):  # quantised without rotation
        codes, scales, _ = oracle.rotate_quantize(x.double().numpy(), None)
        w[n + "8"], w[n + "_scale"] = torch.from_numpy(codes), torch.from_numpy(scales.astype(np.float32))
    o, lse = gpu_fp8(w, causal)
    Or, Lr = oracle.attention(deq(w, "q"), deq(w, "k"), deq(w, "v"), causal=causal)
    check(o, lse, Or, Lr, f"fp8 max jump causal={causal}")


def test_fp8_full_size_whole_tensor():
    """B=2, Hq=Hkv=16, S=8192, D=128, non-causal, 0.5 % outliers x50, rotated
    and block-quantised: relative RMS over the whole O tensor (all 32 heads,
    every element) and the LSE of every row, against the oracle on the
    dequantised inputs; the oracle runs whole heads on a process pool."""
    from oracle import pool
    cfg = workloads.WORKLOADS["fp8_prefill"]
    w = fp8_inputs(workloads.make_workload("fp8_prefill", seed=0))
    o, lse = gpu_fp8(w, cfg["causal"])
    B, Hq = o.shape[0], o.shape[1]
    heads = [(b, h) for b in range(B) for h in range(Hq)]
    Or, Lr = pool.attention_heads(deq(w, "q"), deq(w, "k"), deq(w, "v"), heads, cfg["causal"], 1.0 / np.sqrt(128))
    Or = Or.reshape(o.shape)
    Lr = Lr.reshape(lse.shape)
    rr, dl = check(o, lse, Or, Lr, "fp8 whole tensor")
    per_head = [rel_rms(o[b, h], Or[b, h]) for b, h in heads]
    assert max(per_head) <= FP8_REL_RMS
    print(f"fp8_prefill, whole tensor (32 heads): relative RMS {rr:.4f} (per head max {max(per_head):.4f}), "
          f"max|dLSE| {dl:.3g}")


@pytest.mark.parametrize("Sq,Sk", [(1000, 1000), (700, 1300), (1300, 700)])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_skewed_roles(Sq, Sk, causal):
    """The FP8 kernel issues the next key tile's scores before it consumes the
    current probabilities, so its warp roles may drift up to a key tile apart.
    With attn_debug_skew_roles the issuing thread pauses after each request
    for scores and the first query tile's softmax before each wait for them:
    the other tile's softmax finishes its next probabilities before the
    issuing thread asks for the current ones, and under the causal mask (the
    first tile stopping a key tile early) the second tile's next scores are
    requested while the first tile still sleeps.  A miscounted barrier phase
    would show as a wait that runs out; the results must be those of the
    oracle, as without the delays."""
    import exact_tiled_attention_15_gb300 as eta
    w = fp8_inputs(workloads.make_fp8_prefill(1, 4, 2, Sq, Sk, 128, seed=Sq * 3 + Sk))
    eta.debug_skew_roles(True)
    try:
        o, lse = gpu_fp8(w, causal)
    finally:
        eta.debug_skew_roles(False)
    Or, Lr = oracle.attention(deq(w, "q"), deq(w, "k"), deq(w, "v"), causal=causal)
    check(o, lse, Or, Lr, f"fp8 skewed {Sq}x{Sk} causal={causal}")
    o2, lse2 = gpu_fp8(w, causal)  # the normal build, same inputs: the same bits
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


@pytest.mark.parametrize("B,Hq,Hkv,S,causal", [(2, 16, 16, 8192, False), (1, 8, 2, 4100, True)])
def test_fp8_skewed_roles_long_sequences_bit_equal(B, Hq, Hkv, S, causal):
    """The skewed-role build over many key tiles per CTA (64 at the FP8
    benchmark size; a causal GQA case whose two Q tiles stop a key tile
    apart): the rings wrap many times while the roles sit as far apart as the
    protocol lets them, and the output must be the normal build's, bit for
    bit (the normal build is compared with the oracle at these sizes by the
    whole-tensor tests)."""
    import exact_tiled_attention_15_gb300 as eta
    w = fp8_inputs(workloads.make_fp8_prefill(B, Hq, Hkv, S, S, 128, seed=S + B))
    o, lse = gpu_fp8(w, causal)
    eta.debug_skew_roles(True)
    try:
        o2, lse2 = gpu_fp8(w, causal)
    finally:
        eta.debug_skew_roles(False)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
