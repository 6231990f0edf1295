"""The work accounting behind every roofline number, pinned to figures the
pages print (tests/golden/page_figures.json)."""
import json
import os

import pytest

from exact_tiled_attention_15_gb300 import accounting as acc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")
ENTRIES = json.load(open(GOLDEN))["entries"]


@pytest.mark.parametrize("e", ENTRIES, ids=[e["quantity"] for e in ENTRIES])
def test_page_figure(e):
    a = e["args"]
    q = e["quantity"]
    if q == "score_matrix_bytes":
        got = acc.score_matrix_bytes(a["S"], a["H"], a["elem_bytes"])
    elif q == "score_entries":
        got = acc.score_matrix_bytes(a["N"], 1, 1)
    elif q == "decode_intensity":
        sl = [1000, 2000, 3000]
        got = acc.decode_flops(sl, a["Hq"], a["D"]) / acc.decode_kv_bytes(sl, a["Hkv"], a["D"])
    elif q == "gqa_cache_shrink":
        got = acc.decode_kv_bytes([100], a["Hq"], 128) / acc.decode_kv_bytes([100], a["Hkv"], 128)
    elif q == "memory_saving_ratio":
        got = acc.memory_saving_ratio(a["S"], a["D"])
    elif q == "causal_saving":
        got = acc.prefill_flops(a["B"], a["Hq"], a["S"], a["S"], a["D"], False) / \
            acc.prefill_flops(a["B"], a["Hq"], a["S"], a["S"], a["D"], True)
    else:
        raise AssertionError(q)
    if "value" in e:
        assert got == pytest.approx(e["value"], rel=1e-12), e["cite"]
    else:
        assert e["value_min"] <= got <= e["value_max"], e["cite"]


def test_benchmark_workloads():
    # 4 x 32 heads x 4096^2 x 128, causal: 549.8 GFLOP
    assert acc.prefill_flops(4, 32, 4096, 4096, 128, True) == pytest.approx(549.755813888e9)
    # decode, seed-0 lengths sum to 299,418: 1.2264 GB of K and V
    assert acc.decode_kv_bytes([299418], 8, 128) == pytest.approx(1.226416128e9)


def test_visible_pairs_exact_count():
    """Brute force over a small grid; square causal is S(S+1)/2 (the 'halved'
    count plus the diagonal); Sq > Sk leaves the first rows empty."""
    import numpy as np
    from exact_tiled_attention_15_gb300 import accounting as acc
    for Sq, Sk in ((1, 1), (5, 5), (3, 9), (9, 3), (128, 1000)):
        rows = np.arange(Sq)[:, None]
        keys = np.arange(Sk)[None, :]
        assert acc.visible_pairs(Sq, Sk, True) == int((keys <= rows + (Sk - Sq)).sum())
        assert acc.visible_pairs(Sq, Sk, False) == Sq * Sk
    assert acc.visible_pairs(4096, 4096, True) == 4096 * 4097 // 2
    assert acc.prefill_flops_exact(2, 3, 7, 7, 16, False) == 4 * 16 * 2 * 3 * 49
