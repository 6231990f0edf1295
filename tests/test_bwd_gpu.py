"""GPU parity of the backward (dQ, dK, dV with recomputation) against the
fp64 oracle.  P and dS enter the tensor-core products as bf16 and the
forward's O is bf16, so each gradient tensor is compared by its relative RMS
error (bound 1e-2) and by the largest error relative to its largest entry
(bound 3e-2)."""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_15_gb300 import workloads

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
REL_RMS = 1e-2
REL_MAX = 3e-2


def check(g, ref, what):
    g = np.asarray(g, dtype=np.float64)
    assert np.isfinite(g).all(), what
    nr = np.linalg.norm(ref)
    if nr == 0:
        assert np.abs(g).max() == 0, what
        return 0.0
    rr = np.linalg.norm(g - ref) / nr
    rm = np.abs(g - ref).max() / np.abs(ref).max()
    assert rr <= REL_RMS and rm <= REL_MAX, f"{what}: rel RMS {rr:.3g}, rel max {rm:.3g}"
    return rr


def run(B, Hq, Hkv, Sq, Sk, causal, seed=0, D=128):
    import exact_tiled_attention_15_gb300 as eta
    w = workloads.make_prefill(B, Hq, Hkv, Sq, Sk, D, seed=seed)
    do = workloads.to_bf16(np.random.default_rng(seed + 100).standard_normal((B, Hq, Sq, D)).astype(np.float32))
    q, k, v, dod = w["q"].to(DEV), w["k"].to(DEV), w["v"].to(DEV), do.to(DEV)
    o, lse = eta.fwd(q, k, v, causal=causal)
    dq, dk, dv = eta.bwd(q, k, v, o, lse, dod, causal=causal)
    assert eta.get_error() == 0
    dqr, dkr, dvr, _, _ = oracle.attention_backward(w["q"].double().numpy(), w["k"].double().numpy(),
                                                    w["v"].double().numpy(), do.double().numpy(), causal=causal)
    tag = f"{Hq}/{Hkv} {Sq}x{Sk} D={D} causal={causal}"
    return (check(dq.double().cpu().numpy(), dqr, "dQ " + tag), check(dk.double().cpu().numpy(), dkr, "dK " + tag),
            check(dv.double().cpu().numpy(), dvr, "dV " + tag))


@pytest.mark.parametrize("S", [128, 200, 384])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_square(S, causal):
    run(1, 2, 2, S, S, causal, seed=S)


@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (4, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_gqa(Hq, Hkv, causal):
    run(2, Hq, Hkv, 256, 256, causal, seed=Hq * 3 + Hkv)


@pytest.mark.parametrize("Sq,Sk", [(100, 300), (300, 100)])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_unequal(Sq, Sk, causal):
    """With Sq > Sk causal, the first rows see no key (zero gradients), and key
    tiles no query sees get zero dK, dV."""
    run(1, 2, 1, Sq, Sk, causal, seed=Sq + Sk)


@pytest.mark.parametrize("Hq,Hkv,Sq,Sk", [(2, 2, 384, 384), (4, 1, 200, 330), (2, 1, 300, 100)])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_d64(Hq, Hkv, Sq, Sk, causal):
    """Head dimension 64: one 64-column box per tile; dQ read out of TMEM in one
    piece and staged as two 32-column boxes (over the item's Q and dO tiles)."""
    run(1, Hq, Hkv, Sq, Sk, causal, seed=Sq + 7 * Hq + Hkv, D=64)


def test_bwd_train_workload_whole_tensor():
    """The training workload (B = 4, 32/32 heads, S = 4096, D = 128, causal),
    dO ~ N(0, 1) as in the bench: every element of dQ, dK and dV against the
    oracle, which runs each (batch, head) unit on a process pool; the bounds
    hold for every head and for the whole tensors."""
    import exact_tiled_attention_15_gb300 as eta
    from oracle import pool
    w = workloads.make_workload("train_prefill_mha", seed=0)
    rng = np.random.default_rng(7)
    do = workloads.to_bf16(rng.standard_normal(tuple(w["q"].shape)).astype(np.float32))
    q, k, v, dod = w["q"].to(DEV), w["k"].to(DEV), w["v"].to(DEV), do.to(DEV)
    o, lse = eta.fwd(q, k, v, causal=True)
    dq, dk, dv = eta.bwd(q, k, v, o, lse, dod, causal=True)
    assert eta.get_error() == 0
    B, H = q.shape[0], q.shape[1]
    units = [(b, h) for b in range(B) for h in range(H)]
    dqr, dkr, dvr = pool.backward_units(w["q"].float().numpy(), w["k"].float().numpy(), w["v"].float().numpy(),
                                        do.float().numpy(), units, causal=True)
    g = {"dQ": dq.double().cpu().numpy(), "dK": dk.double().cpu().numpy(), "dV": dv.double().cpu().numpy()}
    r = {"dQ": dqr[:, 0].reshape(g["dQ"].shape), "dK": dkr.reshape(g["dK"].shape), "dV": dvr.reshape(g["dV"].shape)}
    worst = {}
    for name in ("dQ", "dK", "dV"):
        check(g[name], r[name], f"{name} whole tensor")
        worst[name] = max(check(g[name][b, h], r[name][b, h], f"{name} b{b} h{h}") for b, h in units)
    print("backward, whole tensors (128 heads): per-head relative RMS at most "
          + ", ".join(f"{n} {x:.4f}" for n, x in worst.items()))


def test_bwd_more_than_65535_head_pairs():
    """66,000 (batch, KV head) pairs: the backward's grid (key tile, batch, KV
    head) and its pre / post passes are one-dimensional; sampled heads at both
    ends and in the middle against the oracle."""
    import exact_tiled_attention_15_gb300 as eta
    B, H, S, D = 2, 33000, 16, 64
    w = workloads.make_prefill(B, H, H, S, S, D, seed=25)
    do = workloads.to_bf16(np.random.default_rng(26).standard_normal((B, H, S, D)).astype(np.float32))
    q, k, v = (w[n].to(DEV) for n in ("q", "k", "v"))
    o, lse = eta.fwd(q, k, v, causal=True)
    dq, dk, dv = eta.bwd(q, k, v, o, lse, do.to(DEV), causal=True)
    assert eta.get_error() == 0
    for b, h0 in ((0, 0), (1, 16496), (1, H - 8)):
        part = [w[n][b:b + 1, h0:h0 + 8].double().numpy() for n in ("q", "k", "v")]
        refs = oracle.attention_backward(*part, do[b:b + 1, h0:h0 + 8].double().numpy(), causal=True)[:3]
        for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), refs):
            check(g[b:b + 1, h0:h0 + 8].double().cpu().numpy(), r, f"{name} 2x33000 heads b{b} h{h0}")
