"""GPU parity of the host-buffer forward (attn_fwd_host): chunked copies and
kernels on three streams must give exactly the device forward's result, for
one chunk and for several (with a short last chunk and reused buffers), for
pinned and pageable host memory, and match the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_15_gb300 import workloads
from parity import check_bf16

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def run(B, Hq, Hkv, S, D, causal, pinned=True, seed=0):
    import exact_tiled_attention_15_gb300 as eta
    w = workloads.make_prefill(B, Hq, Hkv, S, S, D, seed=seed)
    hq, hk, hv = (w[n].pin_memory() if pinned else w[n].clone() for n in ("q", "k", "v"))
    o_h, l_h = eta.fwd_host(hq, hk, hv, causal=causal, device=DEV)
    torch.cuda.synchronize(DEV)
    assert eta.get_error() == 0
    o_d, l_d = eta.fwd(hq.to(DEV), hk.to(DEV), hv.to(DEV), causal=causal)
    torch.cuda.synchronize(DEV)
    # the same kernel on the same heads: bit-for-bit
    assert torch.equal(o_h, o_d.cpu())
    assert torch.equal(l_h, l_d.cpu())
    return w, o_h, l_h


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv,D", [(4, 4, 128), (8, 2, 128), (4, 1, 64)])
def test_host_small_matches_device_and_oracle(Hq, Hkv, D, causal):
    w, o_h, l_h = run(2, Hq, Hkv, 300, D, causal, seed=Hq + D)
    O, L = oracle.attention(w["q"].double().numpy(), w["k"].double().numpy(), w["v"].double().numpy(),
                            causal=causal)
    check_bf16(o_h.double().numpy(), O, l_h.double().numpy(), L, what=f"fwd_host {Hq}/{Hkv} D{D}")


@pytest.mark.parametrize("pinned", [True, False])
def test_host_many_chunks(pinned):
    """B=2, H=32, S=4096: 64 units in chunks of 19 -> four chunks, the last
    one short, buffer 0 reused by chunk 3."""
    import exact_tiled_attention_15_gb300 as eta
    n1 = eta.fwd_host_workspace_bytes(2, 32, 32, 4096, 4096, 128)
    assert n1 < 64 * 3 * 4096 * 128 * 2 * 4  # smaller than staging every unit
    run(2, 32, 32, 4096, 128, True, pinned=pinned, seed=3)


def test_host_without_lse_through_the_c_abi():
    """lse = NULL: the call skips that copy and O is unchanged."""
    import ctypes
    import exact_tiled_attention_15_gb300 as eta
    B, Hq, Hkv, S, D = 1, 8, 2, 700, 128
    w = workloads.make_prefill(B, Hq, Hkv, S, S, D, seed=12)
    hq, hk, hv = (w[n].pin_memory() for n in ("q", "k", "v"))
    o = torch.empty(hq.shape, dtype=hq.dtype, pin_memory=True)
    nbytes = eta.fwd_host_workspace_bytes(B, Hq, Hkv, S, S, D)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    st = eta.lib().attn_fwd_host(hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), o.data_ptr(), None, B, Hq, Hkv, S, S,
                                 D, 1, 1.0 / np.sqrt(D), ctypes.c_void_p(ws.data_ptr()), nbytes,
                                 ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream))
    assert st == 0
    torch.cuda.synchronize(DEV)
    assert eta.get_error() == 0
    o_d, _ = eta.fwd(hq.to(DEV), hk.to(DEV), hv.to(DEV), causal=True)
    assert torch.equal(o, o_d.cpu())
