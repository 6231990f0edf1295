"""GPU parity of the multi-token decode (T query tokens per sequence against
its cache, bottom-right causal) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_15_gb300 import workloads
from parity import check_bf16

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def run_case(B, Hq, Hkv, T, D, Lmin, Lmax, causal=True, seed=0, seqlens=None, rows=None):
    import exact_tiled_attention_15_gb300 as eta
    w = workloads.make_decode(B, Hq, Hkv, D, Lmin, Lmax, seed=seed, seqlens=seqlens, T=T)
    t = {n: w[n].to(DEV) for n in ("q", "kcache", "vcache", "seqlens")}
    o, lse = eta.decode_multi(t["q"], t["kcache"], t["vcache"], t["seqlens"], causal=causal)
    assert eta.get_error() == 0
    o = o.double().cpu().numpy()
    lse = lse.cpu().numpy()
    sel = list(range(B)) if rows is None else rows
    for i in range(0, len(sel), 8):  # eight sequences at a time bound the fp64 copies of the cache
        s = sel[i:i + 8]
        Or, Lr = oracle.decode_multi(w["q"][s].double().numpy(), w["kcache"][s].double().numpy(),
                                     w["vcache"][s].double().numpy(), w["seqlens"][s].numpy(), causal=causal)
        check_bf16(o[s], Or, lse[s], Lr, what=f"multi decode T={T} {Hq}/{Hkv} causal={causal} b={s[0]}..")


@pytest.mark.parametrize("T", [1, 2, 4, 5, 8, 16])
@pytest.mark.parametrize("causal", [True, False])
def test_multi_tokens(T, causal):
    run_case(B=3, Hq=8, Hkv=2, T=T, D=128, Lmin=20, Lmax=500, causal=causal, seed=T)


@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (8, 1, 64), (4, 4, 128)])
def test_multi_groups(Hq, Hkv, D):
    run_case(B=2, Hq=Hq, Hkv=Hkv, T=4, D=D, Lmin=100, Lmax=900, seed=Hq + D)


def test_multi_short_caches():
    """Caches shorter than T: the first tokens sit before the cache start and
    see nothing; a zero-length cache gives zeros everywhere."""
    run_case(B=5, Hq=8, Hkv=2, T=8, D=128, Lmin=1, Lmax=80, seed=9, seqlens=[0, 1, 3, 8, 80])


def test_multi_full_size_whole_tensor():
    """64 sequences, 32/8 heads, D=128, lengths in [1024, 8192], 4 tokens per
    sequence (draft length 3 plus one): every sequence checked in full."""
    run_case(B=64, Hq=32, Hkv=8, T=4, D=128, Lmin=1024, Lmax=8192, seed=0)
