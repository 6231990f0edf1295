"""Pins of the CPU fp64 oracle against what the pages and the mathematics fix.

Each test is chosen so that a plausible slip in the oracle (a dropped rescale,
a transposed operand, a wrong scale, a wrong GQA index, an off-by-one causal
mask, a sign error in a codec) fails at least one of them.  All run on the CPU.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from exact_tiled_attention_15_gb300 import workloads

TOL = 1e-12


def rand(*shape, seed=0, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# ---------------------------------------------------------------- definition pins
def test_identity_values_recover_softmax_rows():
    """With V = I the output is P itself: rows are non-negative, sum to 1
    ("each row sums to 1", Fast Inference §6.21) and P_ij / P_i0 equals
    exp(scale * q_i.(k_j - k_0)) -- which fixes the scale and the operand order."""
    Sq, Sk, D = 5, 9, 4
    q, k = rand(1, 1, Sq, D, seed=1), rand(1, 1, Sk, D, seed=2)
    v = np.eye(Sk)[None, None]
    scale = 0.37
    O, L = oracle.attention(q, k, v, scale=scale)
    P = O[0, 0]
    assert (P >= 0).all()
    np.testing.assert_allclose(P.sum(1), 1.0, atol=TOL)
    ratio = np.log(P / P[:, :1])
    expect = scale * (q[0, 0] @ (k[0, 0] - k[0, 0, :1]).T)
    np.testing.assert_allclose(ratio, expect, atol=1e-10)
    # LSE makes exp(s_ij - LSE_i) sum to one
    s = scale * q[0, 0] @ k[0, 0].T
    np.testing.assert_allclose(np.exp(s - L[0, 0][:, None]).sum(1), 1.0, atol=TOL)


def test_constant_values_give_constant_output():
    """O is a convex combination of V rows, so V = c everywhere gives O = c."""
    q, k = rand(2, 3, 17, 8, seed=3), rand(2, 3, 23, 8, seed=4)
    v = np.full((2, 3, 23, 8), 2.5)
    for causal in (False, True):
        O, _ = oracle.attention(q, k, v, causal=causal)
        np.testing.assert_allclose(O, 2.5, atol=TOL)


def test_causal_first_row_is_first_value_row():
    """Causal, Sq = Sk: query 0 sees key 0 only, so O_0 = V_0, LSE_0 = s_00."""
    q, k, v = rand(1, 2, 16, 8, seed=5), rand(1, 2, 16, 8, seed=6), rand(1, 2, 16, 8, seed=7)
    O, L = oracle.attention(q, k, v, causal=True, scale=0.5)
    np.testing.assert_allclose(O[:, :, 0], v[:, :, 0], atol=TOL)
    np.testing.assert_allclose(L[:, :, 0], 0.5 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0]), atol=TOL)
    # and the last row sees every key: equals the non-causal last row
    On, Ln = oracle.attention(q, k, v, causal=False, scale=0.5)
    np.testing.assert_allclose(O[:, :, -1], On[:, :, -1], atol=TOL)
    np.testing.assert_allclose(L[:, :, -1], Ln[:, :, -1], atol=TOL)


def test_causal_brute_force_prefix():
    """Causal row i equals the non-causal result over keys 0..i + (Sk - Sq)."""
    Sq, Sk, D = 6, 10, 4
    q, k, v = rand(1, 1, Sq, D, seed=8), rand(1, 1, Sk, D, seed=9), rand(1, 1, Sk, D, seed=10)
    O, L = oracle.attention(q, k, v, causal=True)
    for i in range(Sq):
        n = i + (Sk - Sq) + 1
        Oi, Li = oracle.attention(q[:, :, i:i + 1], k[:, :, :n], v[:, :, :n], causal=False)
        np.testing.assert_allclose(O[:, :, i], Oi[:, :, 0], atol=TOL)
        np.testing.assert_allclose(L[:, :, i], Li[:, :, 0], atol=TOL)


@pytest.mark.parametrize("form", ["per_step", "deferred"])
@pytest.mark.parametrize("block", [1, 7, 64, 128, 300])
@pytest.mark.parametrize("causal", [False, True])
def test_online_softmax_matches_direct_computation(form, block, causal):
    """The tiled online-softmax recurrence gives the same result for any block
    size, in both the per-step and the deferred form (Hardware Co-Design;
    Week 13 step 2: the block size does not matter)."""
    q, k, v = rand(2, 4, 37, 16, seed=11), rand(2, 2, 300, 16, seed=12), rand(2, 2, 300, 16, seed=13)
    O, L = oracle.attention(q, k, v, causal=causal)
    O2, L2 = oracle.attention_online(q, k, v, causal=causal, block=block, form=form)
    np.testing.assert_allclose(O2, O, rtol=1e-12, atol=TOL)
    np.testing.assert_allclose(L2, L, rtol=1e-12, atol=TOL)


def test_online_softmax_handles_large_logits():
    """Huge logits overflow neither form, and the output goes to V_argmax
    (Week 13, common mistakes)."""
    q, k, v = rand(1, 1, 8, 16, seed=14, scale=1e4), rand(1, 1, 64, 16, seed=15), rand(1, 1, 64, 16, seed=16)
    O, L = oracle.attention(q, k, v)
    assert np.isfinite(O).all() and np.isfinite(L).all()
    s = q[0, 0] @ k[0, 0].T / 4.0
    top = s.argmax(1)
    gap = np.sort(s, 1)[:, -1] - np.sort(s, 1)[:, -2]
    assert (gap > 50).all()
    np.testing.assert_allclose(O[0, 0], v[0, 0][top], atol=1e-12)
    for form in ("per_step", "deferred"):
        O2, L2 = oracle.attention_online(q, k, v, block=5, form=form)
        np.testing.assert_allclose(O2, O, atol=1e-9)
        np.testing.assert_allclose(L2, L, rtol=1e-12)


def test_fully_masked_rows_are_zero_not_nan():
    """Causal with Sq > Sk: the first Sq - Sk rows have no key.  They come out
    as O = 0, LSE = -inf, with no NaN (m = -inf must not give e^(-inf+inf))."""
    q, k, v = rand(1, 1, 12, 8, seed=17), rand(1, 1, 5, 8, seed=18), rand(1, 1, 5, 8, seed=19)
    for fn in (oracle.attention, lambda *a, **kw: oracle.attention_online(*a, block=2, **kw)):
        O, L = fn(q, k, v, causal=True)
        assert not np.isnan(O).any() and not np.isnan(L).any()
        np.testing.assert_array_equal(O[0, 0, :7], 0.0)
        assert np.isneginf(L[0, 0, :7]).all()
        assert np.isfinite(L[0, 0, 7:]).all()
        np.testing.assert_allclose(O[0, 0, 7], v[0, 0, 0], atol=TOL)


def test_gqa_equals_mha_on_repeated_heads():
    """GQA with Hkv < Hq equals MHA on K, V repeated per group (contiguous
    groups, Fast Inference §6.2); Hkv = 1 is MQA; Hkv = Hq is MHA."""
    B, Hq, S, D = 2, 8, 19, 8
    q = rand(B, Hq, S, D, seed=20)
    for Hkv in (8, 4, 2, 1):
        k, v = rand(B, Hkv, S, D, seed=21), rand(B, Hkv, S, D, seed=22)
        g = Hq // Hkv
        kr, vr = np.repeat(k, g, axis=1), np.repeat(v, g, axis=1)
        for causal in (False, True):
            O, L = oracle.attention(q, k, v, causal=causal)
            Om, Lm = oracle.attention(q, kr, vr, causal=causal)
            np.testing.assert_array_equal(O, Om)
            np.testing.assert_array_equal(L, Lm)
    # a head's result depends on its own group's K/V only: perturbing group 1
    # must not move heads of group 0
    k, v = rand(B, 2, S, D, seed=23), rand(B, 2, S, D, seed=24)
    O1, _ = oracle.attention(q, k, v)
    k2 = k.copy()
    k2[:, 1] += rand(B, S, D, seed=99)
    O2, _ = oracle.attention(q, k2, v)
    np.testing.assert_array_equal(O1[:, :4], O2[:, :4])
    assert np.abs(O1[:, 4:] - O2[:, 4:]).max() > 1e-3


def test_closed_forms():
    """Q = 0: uniform weights, O = mean of allowed V rows, LSE = ln(#allowed).
    Sk = 1: O = V_0.  Sk = 2: logistic weights, LSE = logaddexp."""
    Sq, Sk, D = 6, 6, 4
    v = rand(1, 1, Sk, D, seed=25)
    q = np.zeros((1, 1, Sq, D))
    k = rand(1, 1, Sk, D, seed=26)
    O, L = oracle.attention(q, k, v, causal=True)
    for i in range(Sq):
        np.testing.assert_allclose(O[0, 0, i], v[0, 0, :i + 1].mean(0), atol=TOL)
        np.testing.assert_allclose(L[0, 0, i], math.log(i + 1), atol=TOL)
    q1 = rand(1, 1, 3, D, seed=27)
    O, L = oracle.attention(q1, k[:, :, :1], v[:, :, :1])
    np.testing.assert_allclose(O[0, 0], np.repeat(v[0, 0, :1], 3, 0), atol=TOL)
    O, L = oracle.attention(q1, k[:, :, :2], v[:, :, :2], scale=0.8)
    s = 0.8 * q1[0, 0] @ k[0, 0, :2].T
    w0 = 1.0 / (1.0 + np.exp(s[:, 1] - s[:, 0]))
    np.testing.assert_allclose(O[0, 0], w0[:, None] * v[0, 0, 0] + (1 - w0)[:, None] * v[0, 0, 1], atol=TOL)
    np.testing.assert_allclose(L[0, 0], np.logaddexp(s[:, 0], s[:, 1]), atol=TOL)


def test_key_permutation_invariance():
    """Without a mask, permuting keys and values together leaves O unchanged."""
    q, k, v = rand(1, 2, 9, 8, seed=28), rand(1, 2, 31, 8, seed=29), rand(1, 2, 31, 8, seed=30)
    perm = np.random.default_rng(31).permutation(31)
    O, L = oracle.attention(q, k, v)
    O2, L2 = oracle.attention(q, k[:, :, perm], v[:, :, perm])
    np.testing.assert_allclose(O2, O, atol=TOL)
    np.testing.assert_allclose(L2, L, atol=TOL)


def test_split_merge_equals_full():
    """Attention over disjoint key chunks, merged by log-sum-exp weights, equals
    attention over all keys (the merge a split-K decode uses)."""
    q, k, v = rand(2, 4, 3, 16, seed=32), rand(2, 4, 200, 16, seed=33), rand(2, 4, 200, 16, seed=34)
    O, L = oracle.attention(q, k, v)
    cuts = [0, 1, 50, 51, 133, 200]
    parts = [oracle.attention(q, k[:, :, a:b], v[:, :, a:b]) for a, b in zip(cuts[:-1], cuts[1:])]
    Om, Lm = oracle.merge_partials([p[0] for p in parts], [p[1] for p in parts])
    np.testing.assert_allclose(Om, O, atol=TOL)
    np.testing.assert_allclose(Lm, L, atol=TOL)
    # an empty chunk (lse = -inf) changes nothing
    Oe, Le = oracle.merge_partials([parts[0][0], np.zeros_like(O)], [parts[0][1], np.full_like(L, -np.inf)])
    np.testing.assert_allclose(Oe, parts[0][0], atol=TOL)
    np.testing.assert_allclose(Le, parts[0][1], atol=TOL)


@pytest.mark.parametrize("Hq,Hkv,Sq,Sk,causal", [(4, 4, 33, 33, False), (4, 4, 33, 33, True),
                                                 (8, 2, 20, 57, False), (6, 1, 40, 40, True)])
def test_matches_library_sdpa(Hq, Hkv, Sq, Sk, causal):
    """Library special case: PyTorch's CPU scaled_dot_product_attention in
    float64 (test only; the oracle does not use it).  Its logsumexp comes
    from the CPU flash kernel, which aligns the causal mask at the top left,
    so LSE is compared where the two alignments coincide (Sq = Sk)."""
    q, k, v = rand(2, Hq, Sq, 16, seed=35), rand(2, Hkv, Sk, 16, seed=36), rand(2, Hkv, Sk, 16, seed=37)
    O, L = oracle.attention(q, k, v, causal=causal)
    tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
    Ot = F.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, enable_gqa=True)
    if not causal or Sq == Sk:
        np.testing.assert_allclose(O, Ot.numpy(), atol=1e-10)
        g = Hq // Hkv
        _, lse = torch.ops.aten._scaled_dot_product_flash_attention_for_cpu(
            tq, tk.repeat_interleave(g, 1), tv.repeat_interleave(g, 1), 0.0, causal)
        np.testing.assert_allclose(L, lse.numpy(), atol=1e-10)


def test_decode_matches_prefill_definition_and_ignores_tail():
    """Decode is the Sq = 1 case over the first seqlens[b] cache rows; rows
    beyond a sequence's length (NaN here) never reach the result."""
    w = workloads.make_decode(B=3, Hq=8, Hkv=2, D=16, Lmin=1, Lmax=40, seed=3)
    q = w["q"].double().numpy()
    kc, vc = w["kcache"].double().numpy(), w["vcache"].double().numpy()
    sl = w["seqlens"].numpy()
    assert np.isnan(kc).any()
    O, L = oracle.decode(q, kc, vc, sl)
    assert np.isfinite(O).all() and np.isfinite(L).all()
    for b in range(3):
        n = sl[b]
        Ob, Lb = oracle.attention(q[b:b + 1, :, None], kc[b:b + 1, :, :n], vc[b:b + 1, :, :n])
        np.testing.assert_allclose(O[b], Ob[0, :, 0], atol=TOL)
        np.testing.assert_allclose(L[b], Lb[0, :, 0], atol=TOL)
        tq = torch.from_numpy(q[b:b + 1, :, None])
        Ot = F.scaled_dot_product_attention(tq, torch.from_numpy(kc[b:b + 1, :, :n]),
                                            torch.from_numpy(vc[b:b + 1, :, :n]), enable_gqa=True)
        np.testing.assert_allclose(O[b], Ot[0, :, 0].numpy(), atol=1e-10)
    # empty sequence
    O0, L0 = oracle.decode(q[:1], kc[:1], vc[:1], np.array([0]))
    assert (O0 == 0).all() and np.isneginf(L0).all()


def test_paged_decode_gathers_pages_in_position_order():
    """Paged decode equals decode on the contiguous cache the pages were filled
    from, for page sizes below, equal to and above the 64-key kernel stage;
    the NaN-poisoned unused rows and spare pages never reach the result."""
    for ps in (16, 64, 128):
        w = workloads.make_paged_decode(B=3, Hq=8, Hkv=2, D=16, Lmin=1, Lmax=300, page_size=ps, seed=ps)
        q = w["q"].double().numpy()
        O, L = oracle.decode_paged(q, w["k_pages"].double().numpy(), w["v_pages"].double().numpy(),
                                   w["block_table"].numpy(), w["seqlens"].numpy(), ps)
        Oc, Lc = oracle.decode(q, w["kcache"].double().numpy(), w["vcache"].double().numpy(), w["seqlens"].numpy())
        assert np.isfinite(O).all()
        np.testing.assert_array_equal(O, Oc)
        np.testing.assert_array_equal(L, Lc)
        # the table really is scrambled
        assert not np.array_equal(np.sort(w["block_table"].numpy().ravel()), w["block_table"].numpy().ravel())


def test_multi_token_decode():
    """T = 1 is decode; with the causal mask the last token sees the whole
    cache and token t sees exactly the first L - T + t + 1 keys (brute force);
    a token before the cache start sees nothing."""
    w1 = workloads.make_decode(B=3, Hq=8, Hkv=2, D=16, Lmin=5, Lmax=60, seed=41, T=1)
    q1 = w1["q"].double().numpy()
    kc, vc, sl = w1["kcache"].double().numpy(), w1["vcache"].double().numpy(), w1["seqlens"].numpy()
    O1, L1 = oracle.decode_multi(q1, kc, vc, sl)
    Od, Ld = oracle.decode(q1[:, :, 0], kc, vc, sl)
    np.testing.assert_allclose(O1[:, :, 0], Od, atol=TOL)
    np.testing.assert_allclose(L1[:, :, 0], Ld, atol=TOL)
    w = workloads.make_decode(B=3, Hq=8, Hkv=2, D=16, Lmin=2, Lmax=60, seed=42, T=5, seqlens=[2, 17, 60])
    q = w["q"].double().numpy()
    kc, vc, sl = w["kcache"].double().numpy(), w["vcache"].double().numpy(), w["seqlens"].numpy()
    O, L = oracle.decode_multi(q, kc, vc, sl, causal=True)
    On, Ln = oracle.decode_multi(q, kc, vc, sl, causal=False)
    np.testing.assert_allclose(O[:, :, -1], On[:, :, -1], atol=TOL)
    for b in range(3):
        for t in range(5):
            n = int(sl[b]) - 5 + t + 1
            if n <= 0:
                assert (O[b, :, t] == 0).all() and np.isneginf(L[b, :, t]).all()
                continue
            Ob, Lb = oracle.decode(q[b:b + 1, :, t], kc[b:b + 1, :, :n], vc[b:b + 1, :, :n], np.array([n]))
            np.testing.assert_allclose(O[b, :, t], Ob[0], atol=TOL)
            np.testing.assert_allclose(L[b, :, t], Lb[0], atol=TOL)


def _loss(q, k, v, do, causal, scale):
    O, _ = oracle.attention(q, k, v, causal=causal, scale=scale)
    return float((O * do).sum())


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_finite_differences(causal):
    """Central differences of sum(dO o O) in float64 pin every gradient entry
    of a tiny GQA case (2 query heads on 1 KV head, Sq != Sk)."""
    q, k, v = rand(1, 2, 4, 3, seed=50), rand(1, 1, 6, 3, seed=51), rand(1, 1, 6, 3, seed=52)
    do = rand(1, 2, 4, 3, seed=53)
    dq, dk, dv, _, _ = oracle.attention_backward(q, k, v, do, causal=causal, scale=0.7)
    h = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = [xp if y is x else y for y in (q, k, v)]
            args_m = [xm if y is x else y for y in (q, k, v)]
            num[idx] = (_loss(*args_p, do, causal, 0.7) - _loss(*args_m, do, causal, 0.7)) / (2 * h)
        np.testing.assert_allclose(g, num, atol=1e-7, rtol=1e-6)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_library_autograd(causal):
    """PyTorch's CPU fp64 autograd through scaled_dot_product_attention (test
    only), with grouped-query heads."""
    q, k, v = rand(2, 4, 33, 16, seed=54), rand(2, 2, 33, 16, seed=55), rand(2, 2, 33, 16, seed=56)
    do = rand(2, 4, 33, 16, seed=57)
    dq, dk, dv, _, _ = oracle.attention_backward(q, k, v, do, causal=causal)
    tq, tk, tv = (torch.from_numpy(x).requires_grad_() for x in (q, k, v))
    F.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, enable_gqa=True).backward(torch.from_numpy(do))
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-10)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-10)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-10)


def test_backward_gqa_is_group_sum_of_mha():
    q = rand(1, 4, 20, 8, seed=58)
    k, v = rand(1, 2, 20, 8, seed=59), rand(1, 2, 20, 8, seed=60)
    do = rand(1, 4, 20, 8, seed=61)
    dq, dk, dv, _, _ = oracle.attention_backward(q, k, v, do, causal=True)
    dq2, dk2, dv2, _, _ = oracle.attention_backward(q, np.repeat(k, 2, 1), np.repeat(v, 2, 1), do, causal=True)
    np.testing.assert_allclose(dq, dq2, atol=TOL)
    np.testing.assert_allclose(dk, dk2.reshape(1, 2, 2, 20, 8).sum(2), atol=TOL)
    np.testing.assert_allclose(dv, dv2.reshape(1, 2, 2, 20, 8).sum(2), atol=TOL)


# ---------------------------------------------------------------- codecs
def test_bf16_decoder_matches_library_cast():
    codes = np.arange(1 << 16, dtype=np.uint16)
    ours = oracle.bf16_decode(codes)
    lib = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(lib))
    ok = ~np.isnan(ours)
    np.testing.assert_array_equal(ours[ok], lib[ok])


def test_e4m3_decoder_matches_library_cast_and_spec_points():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(lib))
    ok = ~np.isnan(ours)
    np.testing.assert_array_equal(ours[ok], lib[ok])
    assert ours[0x7E] == 448.0 and ours[0xFE] == -448.0          # largest finite
    assert ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6    # smallest subnormal / normal
    assert ours[0x38] == 1.0 and np.isnan(ours[0x7F]) and np.isnan(ours[0xFF])
    assert np.isnan(ours).sum() == 2                             # no infinities, two NaNs


def test_dequantize_tiles_matches_library_and_scale_layout():
    from parity import fp8_inputs
    w = fp8_inputs(workloads.make_fp8_prefill(B=1, Hq=2, Hkv=2, Sq=300, Sk=300, D=128, seed=4))
    codes, scales = w["q8"], w["q_scale"]
    assert scales.shape == (1, 2, 3, 1)
    ours = oracle.dequantize_tiles(codes.numpy(), scales.numpy())
    lib = codes.view(torch.float8_e4m3fn).double()
    lib = lib * scales.double().repeat_interleave(128, 2)[:, :, :300].repeat_interleave(128, 3)[..., :128]
    np.testing.assert_array_equal(ours, lib.numpy())
    # each tile's largest magnitude lands on the top code (amax / scale = 448)
    for t in range(3):
        blk = np.abs(oracle.e4m3_decode(codes[0, 0, t * 128:(t + 1) * 128].numpy()))
        assert blk.max() == 448.0


def test_e4m3_encoder_matches_library_cast_including_ties():
    decoded = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))       # +0 .. 448
    mids = (decoded[:-1] + decoded[1:]) / 2                              # exact ties
    rng = np.random.default_rng(43)
    vals = np.concatenate([decoded, mids, -mids, rng.uniform(-448, 448, 20000), rng.normal(0, 1e-2, 5000),
                           [448.0, -448.0, 0.0]])
    ours = oracle.e4m3_encode(vals)
    lib = torch.from_numpy(vals.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # torch rounds from float32; every value above is exact in float32
    np.testing.assert_array_equal(ours, lib)
    np.testing.assert_array_equal(oracle.e4m3_decode(oracle.e4m3_encode(decoded)), decoded)
    assert oracle.e4m3_encode([1e6])[0] == 0x7E and oracle.e4m3_encode([-1e6])[0] == 0xFE   # saturate


def test_rotate_quantize_round_trip_and_tile_scales():
    rng = np.random.default_rng(44)
    x = rng.standard_normal((1, 2, 300, 128))
    x[0, 0, 5, 7] = 40.0                                                  # an outlier
    signs = rng.integers(0, 2, 128) * 2.0 - 1.0
    codes, scales, y = oracle.rotate_quantize(x, signs)
    assert scales.shape == (1, 2, 3, 1)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-12)  # orthogonal
    deq = oracle.dequantize_tiles(codes, scales)
    R = oracle.quant.hadamard(128) * signs[None, :] / np.sqrt(128)
    back = deq @ R.T
    assert np.linalg.norm(back - x) / np.linalg.norm(x) < 0.04          # e4m3 keeps ~3 significant bits
    for t in range(3):                                                    # each tile's largest |y| -> 448
        assert np.abs(oracle.e4m3_decode(codes[0, 0, t * 128:(t + 1) * 128])).max() == 448.0
    # the rotation spreads the outlier over the row: the tile's largest magnitude drops
    c0, s0, _ = oracle.rotate_quantize(x, None)
    assert np.abs(y[0, 0, :128]).max() < 0.5 * np.abs(x[0, 0, :128]).max()
    assert scales[0, 0, 0, 0] < 0.5 * s0[0, 0, 0, 0]
    np.testing.assert_array_equal(c0, oracle.e4m3_encode(x / np.repeat(s0, 128, 2)[:, :, :300]))


def test_rotation_is_orthogonal_and_preserves_scores():
    """Incoherent processing (FlashAttention-3): rotating Q and K by the same
    orthogonal R = H_D diag(s) / sqrt(D) leaves Q K^T unchanged."""
    signs = np.random.default_rng(0).integers(0, 2, 128) * 2.0 - 1.0
    R = oracle.quant.hadamard(128) * signs[None, :] / np.sqrt(128)
    np.testing.assert_allclose(R @ R.T, np.eye(128), atol=1e-12)
    q, k = rand(50, 128, seed=38), rand(60, 128, seed=39)
    np.testing.assert_allclose((q @ R) @ (k @ R).T, q @ k.T, atol=1e-10)
    H = oracle.quant.hadamard(8)
    np.testing.assert_array_equal(H @ H.T, 8 * np.eye(8))
    _, _, y = oracle.rotate_quantize(np.stack([q, q])[None], signs)      # the same R inside rotate_quantize
    np.testing.assert_allclose(y[0, 0], q @ R, atol=1e-12)


# ---------------------------------------------------------------- input generator pins
def test_fp8_draws_recipe():
    """The FP8 draws: bf16 Q, K, V with about 0.5 % of the entries x50, and
    D rotation signs of +-1; nothing is rotated or quantised here."""
    w = workloads.make_fp8_prefill(B=1, Hq=2, Hkv=1, Sq=512, Sk=512, D=128, seed=0)
    assert w["q"].dtype == torch.bfloat16 and w["q"].shape == (1, 2, 512, 128) and w["k"].shape == (1, 1, 512, 128)
    assert set(np.unique(w["signs"])) == {-1.0, 1.0} and w["signs"].shape == (128,)
    big = (w["q"].float().abs() > 8).float().mean().item()     # |N(0,1)| > 8 never happens without a x50
    assert 0.002 < big < 0.008


def test_decode_seqlens_recipe():
    """Seed-0 decode workload: 64 lengths in [1024, 8192]; their sum fixes the
    algorithmic KV bytes of the benchmark."""
    rng = np.random.default_rng(0)
    sl = rng.integers(1024, 8193, size=64)
    assert sl.min() >= 1024 and sl.max() <= 8192
    assert int(sl.sum()) == 299418


# ---------------------------------------------------------------- rotation convention and row blocks
def _popcount(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=np.int64)
    c = np.zeros_like(x)
    while x.any():
        c += x & 1
        x = x >> 1
    return c


@pytest.mark.parametrize("n", [2, 4, 8, 16, 32, 64, 128])
def test_hadamard_is_sylvester_closed_form(n):
    """Sylvester's construction has the closed form H[i, j] = (-1)^popcount(i & j)
    (the bits of i and j, one factor [[1, 1], [1, -1]] per bit).  This fixes the
    order of the blocks: a matrix built as [[H, H], [-H, H]] is also orthogonal
    and fails here."""
    i, j = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    expect = np.where(_popcount(i & j) % 2 == 0, 1.0, -1.0)
    np.testing.assert_array_equal(oracle.quant.hadamard(n), expect)


@pytest.mark.parametrize("D", [64, 128])
def test_rotation_acts_as_hadamard_then_column_signs(D):
    """The rotation is y = x H_D diag(s) / sqrt(D): the unit row e_i goes to
    s_j (-1)^popcount(i & j) / sqrt(D) in column j.  Signs applied to the rows
    instead (diag(s) H) would give s_i (...) and fail for any non-constant s.
    Every one of the D unit rows is checked (D rows of one tile)."""
    signs = np.random.default_rng(45 + D).integers(0, 2, D) * 2.0 - 1.0
    assert 0 < (signs > 0).sum() < D
    x = np.eye(D)[None, None]                                      # row i = e_i
    _, _, y = oracle.rotate_quantize(x, signs)
    i, j = np.meshgrid(np.arange(D), np.arange(D), indexing="ij")
    expect = signs[None, :] * np.where(_popcount(i & j) % 2 == 0, 1.0, -1.0) / np.sqrt(D)
    np.testing.assert_allclose(y[0, 0], expect, rtol=0, atol=1e-15)
    # the code path: every entry has magnitude 1/sqrt(D), so every code is +-448
    codes, scales, _ = oracle.rotate_quantize(x, signs)
    np.testing.assert_allclose(scales[0, 0, 0, 0], (1 / np.sqrt(D)) / 448.0, rtol=1e-15)
    np.testing.assert_array_equal(oracle.e4m3_decode(codes[0, 0]), 448.0 * np.sign(expect))


@pytest.mark.parametrize("Sq,Sk", [(37, 53), (53, 37), (37, 37)])
@pytest.mark.parametrize("causal", [False, True])
def test_row_blocks_do_not_change_the_result(Sq, Sk, causal):
    """attention() forms complete score rows `row_block` at a time only to bound
    memory.  Any block size gives the same numbers up to the summation order
    the matrix library picks for a different number of rows (~1e-16), including
    the causal offset Sk - Sq and rows with no key when Sq > Sk; a
    block-relative row index in the mask fails here by O(1)."""
    q, k, v = rand(2, 4, Sq, 16, seed=46), rand(2, 2, Sk, 16, seed=47), rand(2, 2, Sk, 16, seed=48)
    O1, L1 = oracle.attention(q, k, v, causal=causal, row_block=10 ** 6)
    for rb in (1, 7, 10, 36):
        O2, L2 = oracle.attention(q, k, v, causal=causal, row_block=rb)
        np.testing.assert_allclose(O2, O1, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(L2, L1, rtol=1e-13, atol=1e-14)
        np.testing.assert_array_equal(np.isneginf(L2), np.isneginf(L1))


def test_default_row_block_beyond_one_block_matches_online_pass():
    """Sq = 1100 > the default block of 1024 rows (the path the long workloads
    take): the plain definition equals the independent online-softmax pass, and
    the causal rows past the first block keep their absolute positions."""
    Sq = Sk = 1100
    q, k, v = rand(1, 2, Sq, 8, seed=49), rand(1, 1, Sk, 8, seed=50), rand(1, 1, Sk, 8, seed=51)
    for causal in (False, True):
        O, L = oracle.attention(q, k, v, causal=causal)
        O2, L2 = oracle.attention_online(q, k, v, causal=causal, block=128)
        np.testing.assert_allclose(O, O2, rtol=1e-12, atol=TOL)
        np.testing.assert_allclose(L, L2, rtol=1e-12, atol=TOL)
    # row 1030 (second block) under the causal mask sees exactly keys 0..1030
    O, L = oracle.attention(q, k, v, causal=True)
    Oi, Li = oracle.attention(q[:, :, 1030:1031], k[:, :, :1031], v[:, :, :1031], causal=False)
    np.testing.assert_allclose(O[:, :, 1030], Oi[:, :, 0], atol=TOL)
    np.testing.assert_allclose(L[:, :, 1030], Li[:, :, 0], atol=TOL)


def test_process_pool_runs_the_same_definition_per_head():
    """oracle.pool fans whole heads over spawned worker processes; it must
    return exactly what the serial definition returns for those heads
    (GQA, causal with Sq != Sk, a subset of heads in any order)."""
    from oracle import pool
    q, k, v = rand(2, 4, 40, 16, seed=52), rand(2, 2, 57, 16, seed=53), rand(2, 2, 57, 16, seed=54)
    O, L = oracle.attention(q, k, v, causal=True, scale=0.3)
    heads = [(1, 3), (0, 0), (0, 2), (1, 1)]
    Op, Lp = pool.attention_heads(q, k, v, heads, causal=True, scale=0.3, workers=2)
    for i, (b, h) in enumerate(heads):
        np.testing.assert_array_equal(Op[i], O[b, h])
        np.testing.assert_array_equal(Lp[i], L[b, h])


def test_process_pool_backward_units_equal_the_serial_definition():
    """oracle.pool.backward_units: each (b, KV head) unit's dQ (its query-head
    group), dK and dV from a spawned worker equal the serial definition's,
    bit for bit (GQA 4/2, causal with Sq != Sk, units in any order)."""
    from oracle import pool
    q, k, v = rand(2, 4, 40, 16, seed=55), rand(2, 2, 57, 16, seed=56), rand(2, 2, 57, 16, seed=57)
    do = rand(2, 4, 40, 16, seed=58)
    dq, dk, dv, _, _ = oracle.attention_backward(q, k, v, do, causal=True, scale=0.3)
    units = [(1, 1), (0, 0), (1, 0)]
    dqp, dkp, dvp = pool.backward_units(q, k, v, do, units, causal=True, scale=0.3, workers=2)
    for i, (b, kv) in enumerate(units):
        np.testing.assert_array_equal(dqp[i], dq[b, 2 * kv:2 * kv + 2])
        np.testing.assert_array_equal(dkp[i], dk[b, kv])
        np.testing.assert_array_equal(dvp[i], dv[b, kv])
