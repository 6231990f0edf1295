"""attn_decode_noalloc: the decode entry point for callers that cannot
allocate device scratch (a custom-op or plugin interface that hands over only
inputs and outputs, or a serving loop that must not call cudaMalloc).  It runs
the same kernels as attn_decode with their scratch in the library's fixed
static device array, so its results must match attn_decode's.

This file is collected last on purpose, and it must pass both on its own in a
fresh process and after every other test (the static array then holds the
previous calls' leftovers, which must not matter).
"""
import ctypes

import numpy as np
import pytest
import torch

from exact_tiled_attention_15_gb300 import workloads
from parity import check_bf16

pytestmark = pytest.mark.gpu
SCRATCH_LIMIT = 6


def _noalloc_call(lib, q, kc, vc, sl, o, lse, scale):
    B, Hq, D = q.shape
    Hkv, Lmax = kc.shape[1], kc.shape[2]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return lib.attn_decode_noalloc(p(q), p(kc), p(vc), p(sl), p(o), p(lse), B, Hq, Hkv, Lmax, D, scale, stream)


def test_noalloc_decode_matches_workspace_decode_twice():
    """Two calls in a row with different sizes and data.  Both entry points run
    the same kernels on the same inputs, so the allocation-free call must give
    the very same bits as attn_decode with its own workspace (a stale value
    left in the shared scratch would show up as a difference), and both must
    match the fp64 oracle within the bf16 bound."""
    import exact_tiled_attention_15_gb300 as eta
    import oracle
    lib = eta.lib()
    dev = torch.device("cuda:0")
    for seed, (B, Hq, Hkv, Lmax) in ((0, (8, 32, 8, 3000)), (1, (5, 16, 2, 700))):
        w = workloads.make_decode(B, Hq, Hkv, 128, 1, Lmax, seed=seed)
        q, kc, vc, sl = (w[n].to(dev) for n in ("q", "kcache", "vcache", "seqlens"))
        scale = 1.0 / np.sqrt(128)
        o_ref, lse_ref = eta.decode(q, kc, vc, sl, scale=scale)      # existing entry point, own workspace
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, Hq), float("nan"), device=dev, dtype=torch.float32)
        assert _noalloc_call(lib, q, kc, vc, sl, o, lse, scale) == 0
        assert eta.get_error() == 0
        assert torch.equal(o, o_ref), f"seed {seed}: O differs from attn_decode"
        assert torch.equal(lse, lse_ref), f"seed {seed}: LSE differs from attn_decode"
        Or, Lr = oracle.decode(w["q"].double().numpy(), w["kcache"].double().numpy(), w["vcache"].double().numpy(),
                               w["seqlens"].numpy(), scale)
        check_bf16(o.double().cpu().numpy(), Or, lse.cpu().numpy(), Lr, what=f"noalloc vs oracle, seed {seed}")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import exact_tiled_attention_15_gb300 as eta
    lib = eta.lib()
    # B=1, 16 query heads on one KV head, a 1M-row cache: ~40 MB of split partials
    assert lib.attn_decode_workspace_bytes(1, 16, 1, 1 << 20, 128) > 16 * 1024 * 1024
    A = ctypes.c_void_p(0x10000)
    st = lib.attn_decode_noalloc(A, A, A, A, A, None, 1, 16, 1, 1 << 20, 128, 0.1, None)
    assert st == SCRATCH_LIMIT
    assert lib.attn_status_str(st) == b"ATTN_ERR_SCRATCH_LIMIT"
