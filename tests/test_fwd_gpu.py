"""GPU parity of the bf16 prefill kernel (tcgen05) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_15_gb300 import workloads
from parity import Bf16Report, check_bf16

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def run(B, Hq, Hkv, Sq, Sk, D, causal, seed=0, scale=None, mult=1.0, k_outlier=0.0):
    import exact_tiled_attention_15_gb300 as eta
    w = workloads.make_prefill(B, Hq, Hkv, Sq, Sk, D, seed=seed, k_outlier_frac=k_outlier, k_outlier_mult=20.0)
    if mult != 1.0:  # larger logits; V keeps its scale so the bound stays comparable
        w = {n: (t.float() * mult).to(torch.bfloat16) if n in ("q", "k") else t for n, t in w.items()}
    q, k, v = (w[n].to(DEV) for n in ("q", "k", "v"))
    o, lse = eta.fwd(q, k, v, causal=causal, scale=scale)
    assert eta.get_error() == 0
    Or, Lr = oracle.attention(w["q"].double().numpy(), w["k"].double().numpy(), w["v"].double().numpy(),
                              causal=causal, scale=scale)
    return check_bf16(o.double().cpu().numpy(), Or, lse.cpu().numpy(), Lr,
                      what=f"fwd B{B} {Hq}/{Hkv} {Sq}x{Sk} D{D} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_tiny_config(causal):
    """B=1, Hq=Hkv=2, S=128, D=64, fp32 N(0,1) draws from seed 0 rounded to bf16."""
    run(1, 2, 2, 128, 128, 64, causal, seed=0)


@pytest.mark.parametrize("S", [1, 100, 128, 129, 255, 256, 257, 600])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_square_shapes(S, D, causal):
    run(1, 2, 2, S, S, D, causal, seed=S + D)


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (4, 1), (6, 3)])
@pytest.mark.parametrize("causal", [False, True])
def test_gqa_mqa(Hq, Hkv, causal):
    run(2, Hq, Hkv, 300, 300, 128, causal, seed=Hq * 10 + Hkv)


@pytest.mark.parametrize("Sq,Sk", [(100, 300), (1, 513), (300, 100), (129, 1000)])
@pytest.mark.parametrize("causal", [False, True])
def test_unequal_lengths(Sq, Sk, causal):
    """Sq != Sk: the causal mask aligns at the bottom right; with Sq > Sk the
    first Sq - Sk rows see no key and must come out as O = 0, LSE = -inf."""
    run(1, 4, 2, Sq, Sk, 128, causal, seed=Sq + Sk)


@pytest.mark.parametrize("causal", [False, True])
def test_large_logits_force_rescales(causal):
    """Q and K x4 (scores 16x larger) make the running max move often, which
    exercises the rescale of the TMEM accumulator."""
    run(1, 2, 2, 700, 700, 128, causal, seed=11, mult=4.0)


@pytest.mark.parametrize("causal", [False, True])
def test_running_max_jump_beyond_exp2_range(causal):
    """Keys of the second and later tiles x60: the running max jumps by far
    more than 126 (log2 units), so the rescale factor of the accumulated O
    underflows to 0 and O must be zeroed, not kept."""
    import exact_tiled_attention_15_gb300 as eta
    w = workloads.make_prefill(1, 2, 2, 400, 400, 128, seed=21)
    k = w["k"].float()
    k[:, :, 128:] *= 60.0
    w["k"] = k.to(torch.bfloat16)
    q, kk, v = (w[n].to(DEV) for n in ("q", "k", "v"))
    o, lse = eta.fwd(q, kk, v, causal=causal)
    assert eta.get_error() == 0
    Or, Lr = oracle.attention(w["q"].double().numpy(), w["k"].double().numpy(), w["v"].double().numpy(),
                              causal=causal)
    assert np.abs(Lr[0, 0, 200:] - Lr[0, 0, 200:].min()).max() > 90  # the jump is really there
    check_bf16(o.double().cpu().numpy(), Or, lse.cpu().numpy(), Lr, what="max jump")


@pytest.mark.parametrize("mult", [3.0, 5.0, 8.0])
@pytest.mark.parametrize("causal", [False, True])
def test_running_max_moderate_jumps(mult, causal):
    """Keys past the first tile scaled by 3, 5 or 8: the row max grows by
    roughly 8 to 40 log2 units after the first tile, so probabilities far
    above 1 are exponentiated against a stale running max (and the largest
    jumps go back over the tile with the new max)."""
    import exact_tiled_attention_15_gb300 as eta
    w = workloads.make_prefill(1, 2, 2, 520, 520, 128, seed=int(mult) + 31)
    k = w["k"].float()
    k[:, :, 128:] *= mult
    w["k"] = k.to(torch.bfloat16)
    q, kk, v = (w[n].to(DEV) for n in ("q", "k", "v"))
    o, lse = eta.fwd(q, kk, v, causal=causal)
    assert eta.get_error() == 0
    Or, Lr = oracle.attention(w["q"].double().numpy(), w["k"].double().numpy(), w["v"].double().numpy(),
                              causal=causal)
    check_bf16(o.double().cpu().numpy(), Or, lse.cpu().numpy(), Lr, what=f"jump x{mult}")


def test_k_outliers():
    run(1, 4, 1, 512, 512, 128, True, seed=12, k_outlier=0.01)


def _whole_tensor(name, heads=None):
    """The forward of a named full-size workload, compared element by element
    with the fp64 oracle over every listed (b, h) (all of them by default);
    the oracle runs whole heads on a process pool."""
    import exact_tiled_attention_15_gb300 as eta
    from oracle import pool
    cfg = workloads.WORKLOADS[name]
    w = workloads.make_workload(name, seed=0)
    q, k, v = (w[n].to(DEV) for n in ("q", "k", "v"))
    o, lse = eta.fwd(q, k, v, causal=cfg["causal"])
    assert eta.get_error() == 0
    o, lse = o.cpu(), lse.cpu()
    del q, k, v
    B, Hq = o.shape[0], o.shape[1]
    heads = heads or [(b, h) for b in range(B) for h in range(Hq)]
    Or, Lr = pool.attention_heads(w["q"].float().numpy(), w["k"].float().numpy(), w["v"].float().numpy(), heads,
                                  cfg["causal"], 1.0 / np.sqrt(o.shape[3]))
    rep = Bf16Report()
    for i, (b, h) in enumerate(heads):
        rep = rep.merge(check_bf16(o[b, h].double().numpy(), Or[i], lse[b, h].numpy(), Lr[i],
                                   what=f"{name} b{b} h{h}"))
    assert rep.n == len(heads) * o.shape[2] * o.shape[3]
    print(f"{name}, whole tensor ({len(heads)} heads): {rep}")
    return rep


def test_train_prefill_full_size_whole_tensor():
    """B=4, 32/32 heads, S=4096, D=128, causal: all 128 heads, every element."""
    _whole_tensor("train_prefill_mha")


def test_long_gqa_prefill_full_size_whole_tensor():
    """B=1, 32/8 heads, S=16384, D=128, causal, 1% of K entries x20: all 32
    heads, every element."""
    _whole_tensor("long_gqa_prefill")


def test_very_long_sequence_sampled():
    """A 65,536-token causal GQA prefill (4 query heads on 1 KV head): 256 query
    blocks per head, 512 key tiles for the last rows; sampled rows against the
    oracle, including the first and last rows and tile edges."""
    import exact_tiled_attention_15_gb300 as eta
    S, D = 65536, 128
    w = workloads.make_prefill(1, 4, 1, S, S, D, seed=9)
    q, k, v = (w[n].to(DEV) for n in ("q", "k", "v"))
    o, lse = eta.fwd(q, k, v, causal=True)
    assert eta.get_error() == 0
    o, lse = o.cpu(), lse.cpu()
    rng = np.random.default_rng(2)
    for h in (0, 3):
        rows = np.unique(np.concatenate([[0, 127, 128, 32767, 32768, S - 129, S - 128, S - 1],
                                         rng.integers(0, S, 8)]))
        Or, Lr = oracle.attention_rows(w["q"].double().numpy(), w["k"].double().numpy(), w["v"].double().numpy(),
                                       0, h, rows, True, 1.0 / np.sqrt(D))
        check_bf16(o[0, h, rows].double().numpy(), Or, lse[0, h, rows].numpy(), Lr, what=f"S=65536 h{h}")


def test_chunked_prefill_full_size_whole_tensor():
    """A 512-token chunk against an 8192-key cache that holds it (B=8, 32/8
    heads, causal aligned at the bottom right): all 256 heads, every element."""
    _whole_tensor("chunked_prefill")


def test_more_than_65535_head_pairs():
    """66,000 (batch, head) pairs, beyond what a 16-bit grid dimension holds: the
    launch folds (query block, batch, head) into grid x.  Head ranges at both
    ends and in the middle of the batch match the oracle."""
    import exact_tiled_attention_15_gb300 as eta
    B, H, S, D = 2, 33000, 16, 64
    w = workloads.make_prefill(B, H, H, S, S, D, seed=23)
    o, lse = eta.fwd(*(w[n].to(DEV) for n in ("q", "k", "v")), causal=True)
    assert eta.get_error() == 0
    for b, h0 in ((0, 0), (1, 16496), (1, H - 8)):
        part = {n: w[n][b:b + 1, h0:h0 + 8].double().numpy() for n in ("q", "k", "v")}
        Or, Lr = oracle.attention(part["q"], part["k"], part["v"], causal=True)
        check_bf16(o[b:b + 1, h0:h0 + 8].double().cpu().numpy(), Or, lse[b:b + 1, h0:h0 + 8].cpu().numpy(), Lr,
                   what=f"fwd 2x33000 heads b{b} h{h0}")
