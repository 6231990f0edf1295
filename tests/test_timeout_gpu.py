"""The bounded waits inside the prefill, backward and quantise pipelines, made
to run out on purpose.

Inside a forward CTA the softmax warps wait for the scores and the tensor-core
issuer waits for the probabilities.  With attn_debug_stall_role_waits the
softmax warps first wait for a signal that nothing gives, and the bound of the
waits between warp roles is 1 ms, so those waits run out (the issuer's wait
for probabilities too): the kernel must record ATTN_ERR_TIMEOUT, let the
copies and products it started complete (those waits keep their normal
bound), free its tensor memory and end.  attn_get_error() then reports the
timeout once, and an ordinary call in the same process afterwards must be
correct -- the GPU context survived.

No GPU is faulted, trapped or hung: every wait ends, the stalled ones after
1 ms.  The sizes keep the K and V rings from ever waiting for a freed slot (at
most two K and three V tiles per CTA), so no wait with the normal 4 s bound is
left waiting on a side that gave up.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_15_gb300 import workloads
from parity import FP8_REL_RMS, check_bf16, fp8_inputs, rel_rms

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
ATTN_ERR_TIMEOUT = 4


def _stalled(fn):
    import exact_tiled_attention_15_gb300 as eta
    assert eta.get_error() == 0
    eta.debug_stall_role_waits(True)
    try:
        fn()
        status = eta.get_error()
    finally:
        eta.debug_stall_role_waits(False)
    return status


@pytest.mark.parametrize("S", [128, 256])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_forward_wait_runs_out_then_next_call_is_correct(S, D, causal):
    import exact_tiled_attention_15_gb300 as eta
    w = workloads.make_prefill(1, 2, 2, S, S, D, seed=S + D)
    q, k, v = (w[n].to(DEV) for n in ("q", "k", "v"))
    st = _stalled(lambda: eta.fwd(q, k, v, causal=causal))
    assert st == ATTN_ERR_TIMEOUT, eta.STATUS.get(st, st)
    assert eta.get_error() == 0  # reported once, then cleared
    o, lse = eta.fwd(q, k, v, causal=causal)
    assert eta.get_error() == 0
    Or, Lr = oracle.attention(w["q"].double().numpy(), w["k"].double().numpy(), w["v"].double().numpy(),
                              causal=causal)
    check_bf16(o.double().cpu().numpy(), Or, lse.cpu().numpy(), Lr, what=f"after timeout S{S} D{D}")


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_wait_runs_out_then_next_call_is_correct(causal):
    """The FP8 instantiation signals differently (one O commit per Q tile, K
    slots handed back with the V slots); two key tiles per CTA and three-stage
    rings, so no producer ever waits for a freed slot."""
    import exact_tiled_attention_15_gb300 as eta
    w = fp8_inputs(workloads.make_fp8_prefill(1, 2, 2, 256, 256, 128, seed=3))
    t = [w[n].to(DEV) for n in ("q8", "k8", "v8", "q_scale", "k_scale", "v_scale")]
    st = _stalled(lambda: eta.fwd_fp8(*t, causal=causal))
    assert st == ATTN_ERR_TIMEOUT, eta.STATUS.get(st, st)
    assert eta.get_error() == 0
    o, lse = eta.fwd_fp8(*t, causal=causal)
    assert eta.get_error() == 0
    deq = [oracle.dequantize_tiles(w[n + "8"].numpy(), w[n + "_scale"].numpy()) for n in ("q", "k", "v")]
    Or, Lr = oracle.attention(*deq, causal=causal)
    assert rel_rms(o.double().cpu().numpy(), Or) <= FP8_REL_RMS
    assert np.abs(lse.cpu().numpy() - Lr).max() <= 1e-3


@pytest.mark.parametrize("causal", [False, True])
def test_backward_wait_runs_out_then_next_call_is_correct(causal):
    """The same for the backward: its gradient warps stall, the tensor-core
    issuer's wait for the probabilities runs out; at most two query tiles per
    key tile (S = 256), so the Q / dO ring never waits for a freed slot."""
    import exact_tiled_attention_15_gb300 as eta
    w = workloads.make_prefill(1, 2, 2, 256, 256, 128, seed=5)
    q, k, v = (w[n].to(DEV) for n in ("q", "k", "v"))
    do = workloads.to_bf16(np.random.default_rng(6).standard_normal((1, 2, 256, 128)).astype(np.float32)).to(DEV)
    o, lse = eta.fwd(q, k, v, causal=causal)
    assert eta.get_error() == 0
    st = _stalled(lambda: eta.bwd(q, k, v, o, lse, do, causal=causal))
    assert st == ATTN_ERR_TIMEOUT, eta.STATUS.get(st, st)
    assert eta.get_error() == 0
    dq, dk, dv = eta.bwd(q, k, v, o, lse, do, causal=causal)
    assert eta.get_error() == 0
    refs = oracle.attention_backward(w["q"].double().numpy(), w["k"].double().numpy(), w["v"].double().numpy(),
                                     do.double().cpu().numpy(), causal=causal)[:3]
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), refs):
        rel = np.linalg.norm(g.double().cpu().numpy() - r) / np.linalg.norm(r)
        assert rel <= 1e-2, f"{name} after timeout: relative RMS {rel:.3g}"


def test_quantise_wait_runs_out_then_next_call_is_correct():
    """The rotate + quantise kernel: its epilogue warps stall, so no product's
    accumulator is ever read out; at most four tiles per CTA, so neither the
    input ring nor the accumulators ever wait for a freed slot."""
    import exact_tiled_attention_15_gb300 as eta
    from test_quant_gpu import check, signs_for
    rng = np.random.default_rng(9)
    x = rng.standard_normal((1, 2, 300, 128)).astype(np.float32)
    x[rng.random(x.shape) < 0.005] *= 50.0
    xb = workloads.to_bf16(x)
    signs = signs_for(9)
    xd, sg = xb.to(DEV), torch.from_numpy(signs.astype(np.float32)).to(DEV)
    st = _stalled(lambda: eta.rotate_quantize_fp8(xd, sg))
    assert st == ATTN_ERR_TIMEOUT, eta.STATUS.get(st, st)
    assert eta.get_error() == 0
    codes, scales = eta.rotate_quantize_fp8(xd, sg)
    assert eta.get_error() == 0
    check(xb, signs, codes.cpu(), scales.cpu(), "after timeout")


@pytest.mark.parametrize("T", [1, 4])
def test_decode_wait_runs_out_then_next_call_is_correct(T):
    """The split decode: its consumer warps stall; each split covers at most a
    few 64-key stages, and a producer that would need a freed stage gives up
    after the same 1 ms, so every wait ends."""
    import exact_tiled_attention_15_gb300 as eta
    w = workloads.make_decode(3, 8, 2, 128, 100, 600, seed=11 + T, T=None if T == 1 else T)
    q, kc, vc, sl = (w[n].to(DEV) for n in ("q", "kcache", "vcache", "seqlens"))
    call = (lambda: eta.decode(q, kc, vc, sl)) if T == 1 else (lambda: eta.decode_multi(q, kc, vc, sl))
    st = _stalled(call)
    assert st == ATTN_ERR_TIMEOUT, eta.STATUS.get(st, st)
    assert eta.get_error() == 0
    o, lse = call()
    assert eta.get_error() == 0
    qn, kn, vn = (w[n].double().numpy() for n in ("q", "kcache", "vcache"))
    if T == 1:
        Or, Lr = oracle.decode(qn, kn, vn, w["seqlens"].numpy(), 1 / np.sqrt(128))
    else:
        Or, Lr = oracle.decode_multi(qn, kn, vn, w["seqlens"].numpy(), causal=True, scale=1 / np.sqrt(128))
    check_bf16(o.double().cpu().numpy(), Or, lse.cpu().numpy(), Lr, what=f"decode T{T} after timeout")
