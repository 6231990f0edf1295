"""GPU parity of the paged-KV decode (block-table gather by TMA) against the
fp64 oracle, which gathers the pages by their definition."""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_15_gb300 import workloads
from parity import check_bf16

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def run_case(B, Hq, Hkv, D, Lmin, Lmax, ps, seed=0, seqlens=None, check_rows=None):
    import exact_tiled_attention_15_gb300 as eta
    w = workloads.make_paged_decode(B, Hq, Hkv, D, Lmin, Lmax, ps, seed=seed, seqlens=seqlens)
    t = {n: w[n].to(DEV) for n in ("q", "k_pages", "v_pages", "block_table", "seqlens")}
    o, lse = eta.decode_paged(t["q"], t["k_pages"], t["v_pages"], t["block_table"], t["seqlens"])
    assert eta.get_error() == 0
    o = o.double().cpu().numpy()
    lse = lse.cpu().numpy()
    rows = range(B) if check_rows is None else check_rows
    kp, vp = w["k_pages"].double().numpy(), w["v_pages"].double().numpy()  # once: the pools are shared
    for b in rows:
        Or, Lr = oracle.decode_paged(w["q"][b:b + 1].double().numpy(), kp, vp, w["block_table"][b:b + 1].numpy(),
                                     w["seqlens"][b:b + 1].numpy(), ps)
        check_bf16(o[b:b + 1], Or, lse[b:b + 1], Lr, what=f"paged decode ps={ps} b={b}")


@pytest.mark.parametrize("ps", [16, 32, 64, 128, 256])
def test_paged_page_sizes(ps):
    run_case(B=4, Hq=8, Hkv=2, D=128, Lmin=1, Lmax=700, ps=ps, seed=ps)


@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (16, 1, 64), (8, 8, 64)])
def test_paged_groups(Hq, Hkv, D):
    run_case(B=3, Hq=Hq, Hkv=Hkv, D=D, Lmin=50, Lmax=400, ps=32, seed=Hq + D)


def test_paged_ragged_edges():
    run_case(B=7, Hq=8, Hkv=2, D=128, Lmin=1, Lmax=640, ps=64, seed=3, seqlens=[0, 1, 63, 64, 65, 129, 640])


def test_paged_full_size_whole_tensor():
    """64 sequences, 32/8 heads, D=128, lengths in [1024, 8192], 64-row pages
    shuffled through the pool: every sequence checked in full."""
    run_case(B=64, Hq=32, Hkv=8, D=128, Lmin=1024, Lmax=8192, ps=64, seed=0)


def test_paged_bad_block_table_entry_is_reported():
    """A live block-table entry outside [0, num_pages) (past the pool, or
    negative): the kernel reads page 0 in its place -- no fault, no read
    outside the pool -- and records ATTN_ERR_BAD_INDEX for attn_get_error;
    the other sequences' results are unaffected, and a later call with a good
    table is clean and correct."""
    import exact_tiled_attention_15_gb300 as eta
    ps = 64
    w = workloads.make_paged_decode(4, 8, 2, 128, 200, 600, ps, seed=31)
    num_pages = w["k_pages"].shape[0]
    t = {n: w[n].to(DEV) for n in ("q", "k_pages", "v_pages", "seqlens")}
    for bad in (num_pages + 5, -1):
        bt = w["block_table"].clone()
        bt[2, 1] = bad  # sequence 2 holds at least 200 rows, so its second page is read
        o, lse = eta.decode_paged(t["q"], t["k_pages"], t["v_pages"], bt.to(DEV), t["seqlens"])
        assert eta.get_error() == eta.ATTN_ERR_BAD_INDEX
        assert eta.get_error() == 0  # reported once
        for b in (0, 1, 3):
            Or, Lr = oracle.decode_paged(w["q"][b:b + 1].double().numpy(), w["k_pages"].double().numpy(),
                                         w["v_pages"].double().numpy(), w["block_table"][b:b + 1].numpy(),
                                         w["seqlens"][b:b + 1].numpy(), ps)
            check_bf16(o[b:b + 1].double().cpu().numpy(), Or, lse[b:b + 1].cpu().numpy(), Lr,
                       what=f"paged decode, bad entry {bad} in sequence 2, b={b}")
    run_case(B=4, Hq=8, Hkv=2, D=128, Lmin=200, Lmax=600, ps=ps, seed=31)
