"""GPU parity of the split-K decode kernel against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_15_gb300 import workloads
from parity import check_bf16

pytestmark = pytest.mark.gpu


def run_case(B, Hq, Hkv, D, Lmin, Lmax, seed=0, seqlens=None, scale=None):
    import exact_tiled_attention_15_gb300 as eta
    w = workloads.make_decode(B, Hq, Hkv, D, Lmin, Lmax, seed=seed, seqlens=seqlens)
    dev = torch.device("cuda:0")
    q, kc, vc, sl = (w[n].to(dev) for n in ("q", "kcache", "vcache", "seqlens"))
    o, lse = eta.decode(q, kc, vc, sl, scale=scale)
    assert eta.get_error() == 0
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    Or, Lr = oracle.decode(w["q"].double().numpy(), w["kcache"].double().numpy(), w["vcache"].double().numpy(),
                           w["seqlens"].numpy(), scale)
    return check_bf16(o.double().cpu().numpy(), Or, lse.cpu().numpy(), Lr, what=f"decode B{B} {Hq}/{Hkv} D{D}")


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 2), (32, 8), (16, 1), (32, 1), (12, 4)])
@pytest.mark.parametrize("D", [64, 128])
def test_decode_group_sizes(Hq, Hkv, D):
    run_case(B=3, Hq=Hq, Hkv=Hkv, D=D, Lmin=1, Lmax=300, seed=Hq + Hkv + D)


def test_decode_ragged_lengths_and_edges():
    # lengths: empty, 1, a tile minus one, exactly a tile, tile + 1, several tiles, Lmax
    sl = [0, 1, 63, 64, 65, 130, 511, 777]
    run_case(B=len(sl), Hq=8, Hkv=2, D=128, Lmin=1, Lmax=777, seed=5, seqlens=sl)


def test_decode_long_cache_many_splits():
    run_case(B=2, Hq=32, Hkv=8, D=128, Lmin=20000, Lmax=20000, seed=6)


def test_decode_large_logits():
    run_case(B=2, Hq=8, Hkv=2, D=128, Lmin=100, Lmax=200, seed=7, scale=3.0)


def test_decode_full_size_whole_tensor():
    """The benchmark workload (64 sequences, 32/8 heads, D=128, lengths in
    [1024, 8192]): every sequence, every head, every element of O and every
    LSE against the oracle."""
    import exact_tiled_attention_15_gb300 as eta
    cfg = workloads.WORKLOADS["gqa_decode"]
    w = workloads.make_decode(cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["Lmin"], cfg["Lmax"], seed=0)
    dev = torch.device("cuda:0")
    q, kc, vc, sl = (w[n].to(dev) for n in ("q", "kcache", "vcache", "seqlens"))
    o, lse = eta.decode(q, kc, vc, sl)
    assert eta.get_error() == 0
    o = o.double().cpu().numpy()
    lse = lse.cpu().numpy()
    assert np.isfinite(o).all()
    for b in range(cfg["B"]):
        n = int(w["seqlens"][b])
        Or, Lr = oracle.decode(w["q"][b:b + 1].double().numpy(), w["kcache"][b:b + 1, :, :n].double().numpy(),
                               w["vcache"][b:b + 1, :, :n].double().numpy(), np.array([n]))
        check_bf16(o[b:b + 1], Or, lse[b:b + 1], Lr, what=f"decode full-size b={b}")


def test_decode_more_than_65535_head_pairs():
    """B * Hkv = 72,000 and B * Hq = 144,000: the split and combine grids are
    one-dimensional; sampled heads at both ends and in the middle against the
    oracle (query heads 2k, 2k + 1 read KV head k)."""
    import exact_tiled_attention_15_gb300 as eta
    B, Hq, Hkv, D = 2, 72000, 36000, 64
    w = workloads.make_decode(B, Hq, Hkv, D, 1, 20, seed=24)
    dev = torch.device("cuda:0")
    o, lse = eta.decode(*(w[n].to(dev) for n in ("q", "kcache", "vcache", "seqlens")))
    assert eta.get_error() == 0
    for b, k0 in ((0, 0), (1, 17996), (1, Hkv - 8)):
        q = w["q"][b:b + 1, 2 * k0:2 * k0 + 16].double().numpy()
        kc = w["kcache"][b:b + 1, k0:k0 + 8].double().numpy()
        vc = w["vcache"][b:b + 1, k0:k0 + 8].double().numpy()
        Or, Lr = oracle.decode(q, kc, vc, w["seqlens"][b:b + 1].numpy(), 1 / np.sqrt(D))
        check_bf16(o[b:b + 1, 2 * k0:2 * k0 + 16].double().cpu().numpy(), Or,
                   lse[b:b + 1, 2 * k0:2 * k0 + 16].cpu().numpy(), Lr, what=f"decode 72000/36000 b{b} kv{k0}")


def test_decode_length_out_of_range_is_reported():
    """seqlens[b] outside [0, Lmax] is clamped into it (Lmax + 7 -> Lmax,
    -3 -> 0: O = 0, LSE = -inf) and recorded as ATTN_ERR_BAD_INDEX for
    attn_get_error; every sequence then matches the oracle at its clamped
    length, and a later call with good lengths is clean."""
    import exact_tiled_attention_15_gb300 as eta
    Lmax = 400
    w = workloads.make_decode(4, 8, 2, 128, 1, Lmax, seed=32, seqlens=[5, Lmax, 300, 0])
    dev = torch.device("cuda:0")
    q, kc, vc = (w[n].to(dev) for n in ("q", "kcache", "vcache"))
    bad = torch.tensor([5, Lmax + 7, 300, -3], dtype=torch.int32, device=dev)
    o, lse = eta.decode(q, kc, vc, bad)
    assert eta.get_error() == eta.ATTN_ERR_BAD_INDEX
    assert eta.get_error() == 0
    Or, Lr = oracle.decode(w["q"].double().numpy(), w["kcache"].double().numpy(), w["vcache"].double().numpy(),
                           w["seqlens"].numpy(), 1 / np.sqrt(128))
    check_bf16(o.double().cpu().numpy(), Or, lse.cpu().numpy(), Lr, what="decode, clamped lengths")
    o, lse = eta.decode(q, kc, vc, w["seqlens"].to(dev))
    assert eta.get_error() == 0
