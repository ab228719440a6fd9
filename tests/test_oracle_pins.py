"""Pins for the fp64 oracle (CPU only).

The oracle is checked against things that do not come from the oracle:
an independent pure-Python brute force, closed forms, invariants that the
mathematics of softmax attention fixes, exact decoders checked against
library conversions, and library routines for the special cases that reduce
to them.  Each test is chosen so that a plausible slip in the oracle (a
dropped scale, a wrong sign, a swapped B/S/H index, a wrong causal offset,
a V/K mix-up, a base-2 LSE) fails at least one of them.
"""
import itertools
import math
import random

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


# --------------------------------------------------------------------------
# an independent brute force: plain Python floats, explicit visible sets
# --------------------------------------------------------------------------
def brute_force(q, k, v, scale, causal):
    """q [B,Sq,H,D], k/v [B,Sk,Hk,D] nested lists -> O [B,Sq,H,Dv], LSE [B,H,Sq].
    Query head h reads key/value head h // (H // Hk)."""
    B, Sq, H = len(q), len(q[0]), len(q[0][0])
    Sk = len(k[0])
    Hk = len(k[0][0]) if Sk else H
    grp = H // Hk
    Dv = len(v[0][0][0]) if Sk else 0
    O = [[[None] * H for _ in range(Sq)] for _ in range(B)]
    L = [[[None] * Sq for _ in range(H)] for _ in range(B)]
    for b in range(B):
        for h in range(H):
            for i in range(Sq):
                vis = [j for j in range(Sk) if (not causal) or (j - i <= Sk - Sq)]
                if not vis:
                    O[b][i][h] = [0.0] * len(v[0][0][0]) if Sk else [0.0]
                    L[b][h][i] = -math.inf
                    continue
                hk = h // grp
                s = {j: scale * sum(a * c for a, c in zip(q[b][i][h], k[b][j][hk])) for j in vis}
                e = {j: math.exp(s[j]) for j in vis}  # tiny values: no overflow
                z = sum(e.values())
                O[b][i][h] = [sum(e[j] * v[b][j][hk][c] for j in vis) / z for c in range(Dv)]
                L[b][h][i] = math.log(z)
    return O, L


def _rand(shape, rng):
    return np.asarray(rng.standard_normal(shape), dtype=np.float64)


@pytest.mark.parametrize("seed", range(16))
def test_brute_force_tiny(seed):
    rng = np.random.default_rng(seed)
    B, H = rng.integers(1, 3), rng.integers(1, 4)
    Hk = H if seed < 10 else 1 if seed % 2 else H  # MHA, and multi-query for some seeds
    if seed >= 12:
        H, Hk = 4, 2                                  # grouped-query: 2 query heads per K/V head
    Sq, Sk = int(rng.integers(1, 9)), int(rng.integers(1, 9))
    D, Dv = int(rng.integers(1, 5)), int(rng.integers(1, 5))
    causal = bool(seed % 2)
    scale = float(rng.uniform(0.2, 1.5))
    q, k, v = _rand((B, Sq, H, D), rng), _rand((B, Sk, Hk, D), rng), _rand((B, Sk, Hk, Dv), rng)
    o, lse = oracle.attention(q, k, v, softmax_scale=scale, causal=causal)
    O, L = brute_force(q.tolist(), k.tolist(), v.tolist(), scale, causal)
    O = np.array(O, dtype=np.float64)
    L = np.array(L, dtype=np.float64)
    fin = np.isfinite(L)
    assert np.array_equal(fin, np.isfinite(lse))
    assert np.allclose(lse[fin], L[fin], rtol=0, atol=1e-12)
    assert np.all(lse[~fin] == -np.inf)
    assert np.allclose(o, O, rtol=0, atol=1e-12)


def test_hand_worked_two_keys():
    # one query q = (1, 0), keys (1,0) and (0,1), scale 1: s = (1, 0)
    # softmax = (e/(e+1), 1/(e+1)); O = softmax . V ; LSE = ln(e + 1)
    q = np.array([[[[1.0, 0.0]]]])
    k = np.array([[[[1.0, 0.0]], [[0.0, 1.0]]]])
    v = np.array([[[[1.0, 2.0]], [[3.0, 4.0]]]])
    o, lse = oracle.attention(q, k, v, softmax_scale=1.0)
    e = math.e
    p0, p1 = e / (e + 1), 1 / (e + 1)
    assert o[0, 0, 0] == pytest.approx([p0 * 1 + p1 * 3, p0 * 2 + p1 * 4], abs=1e-15)
    assert lse[0, 0, 0] == pytest.approx(math.log(e + 1), abs=1e-15)
    # scale 2 and causal (row 0 sees key 0 only when Sq == Sk == 1 ... here Sq=1,Sk=2:
    # bottom-right alignment lets row 0 see keys j <= 0 + 2 - 1 = 1, i.e. both)
    o2, lse2 = oracle.attention(q, k, v, softmax_scale=2.0, causal=True)
    e2 = math.exp(2.0)
    assert lse2[0, 0, 0] == pytest.approx(math.log(e2 + 1), abs=1e-15)
    assert o2[0, 0, 0, 0] == pytest.approx((e2 * 1 + 3) / (e2 + 1), abs=1e-15)


def test_constant_v_returns_that_row():
    rng = np.random.default_rng(1)
    q, k = _rand((2, 7, 3, 5), rng), _rand((2, 9, 3, 5), rng)
    c = rng.standard_normal(4)
    v = np.broadcast_to(c, (2, 9, 3, 4)).copy()
    for causal in (False, True):
        o, _ = oracle.attention(q, k, v, softmax_scale=0.7, causal=causal)
        assert np.allclose(o, np.broadcast_to(c, o.shape), atol=1e-13)


@pytest.mark.parametrize("causal,sq,sk", [(False, 6, 10), (True, 10, 10), (True, 4, 9),
                                          (True, 9, 4)])
def test_zero_q_gives_log_count_and_mean(causal, sq, sk):
    rng = np.random.default_rng(2)
    q = np.zeros((1, sq, 2, 8))
    k, v = _rand((1, sk, 2, 8), rng), _rand((1, sk, 2, 3), rng)
    o, lse = oracle.attention(q, k, v, softmax_scale=0.35, causal=causal)
    for i in range(sq):
        n = sk if not causal else max(0, min(sk, i + sk - sq + 1))
        for h in range(2):
            if n == 0:
                assert lse[0, h, i] == -np.inf and np.all(o[0, i, h] == 0)
            else:
                assert lse[0, h, i] == pytest.approx(math.log(n), abs=1e-13)
                assert np.allclose(o[0, i, h], v[0, :n, h].mean(axis=0), atol=1e-13)


def test_causal_row_zero_is_v0():
    rng = np.random.default_rng(3)
    q, k, v = _rand((2, 12, 2, 6), rng), _rand((2, 12, 2, 6), rng), _rand((2, 12, 2, 6), rng)
    o, lse = oracle.attention(q, k, v, softmax_scale=0.41, causal=True)
    assert np.allclose(o[:, 0], v[:, 0], atol=1e-14)
    s00 = 0.41 * np.einsum("bhd,bhd->bh", q[:, 0], k[:, 0])
    assert np.allclose(lse[:, :, 0], s00, atol=1e-14)


def test_empty_keys_give_zero_and_minus_inf():
    rng = np.random.default_rng(4)
    q = _rand((1, 5, 2, 4), rng)
    k = np.zeros((1, 0, 2, 4))
    v = np.zeros((1, 0, 2, 4))
    o, lse = oracle.attention(q, k, v, softmax_scale=1.0)
    assert np.all(o == 0) and np.all(lse == -np.inf)


def test_probabilities_sum_to_one_and_masked_are_zero():
    rng = np.random.default_rng(5)
    B, Sq, Sk, H = 1, 6, 8, 2
    q, k, v = _rand((B, Sq, H, 4), rng), _rand((B, Sk, H, 4), rng), _rand((B, Sk, H, 4), rng)
    rows = oracle.all_rows(B, H, seqlen_q=Sq)
    o, lse, p = oracle.attention_rows(q, k, v, rows, softmax_scale=0.5, causal=True,
                                      return_probs=True)
    assert np.allclose(p.sum(axis=1), 1.0, atol=1e-14)
    for r, (_, _, i) in enumerate(rows):
        last = i + Sk - Sq
        assert np.all(p[r, last + 1:] == 0) and np.all(p[r, :last + 1] > 0)
    # O is the probability-weighted sum of V rows
    for r, (b, h, i) in enumerate(rows):
        assert np.allclose(o[r], p[r] @ v[b, :, h], atol=1e-14)


def test_permutation_invariance_noncausal():
    rng = np.random.default_rng(6)
    q, k, v = _rand((2, 5, 3, 4), rng), _rand((2, 11, 3, 4), rng), _rand((2, 11, 3, 6), rng)
    o, lse = oracle.attention(q, k, v, softmax_scale=0.8)
    perm = rng.permutation(11)
    o2, lse2 = oracle.attention(q, k[:, perm], v[:, perm], softmax_scale=0.8)
    assert np.allclose(o, o2, atol=1e-13) and np.allclose(lse, lse2, atol=1e-13)


def test_linearity_in_v():
    rng = np.random.default_rng(7)
    q, k, v = _rand((1, 9, 2, 4), rng), _rand((1, 9, 2, 4), rng), _rand((1, 9, 2, 4), rng)
    a, b = -1.7, 0.3
    for causal in (False, True):
        o, _ = oracle.attention(q, k, v, softmax_scale=0.6, causal=causal)
        o2, _ = oracle.attention(q, k, a * v + b, softmax_scale=0.6, causal=causal)
        assert np.allclose(o2, a * o + b, atol=1e-13)


def test_key_shift_moves_lse_only():
    rng = np.random.default_rng(8)
    q, k, v = _rand((1, 7, 2, 5), rng), _rand((1, 7, 2, 5), rng), _rand((1, 7, 2, 5), rng)
    c = rng.standard_normal(5)
    scale = 0.9
    for causal in (False, True):
        o, lse = oracle.attention(q, k, v, softmax_scale=scale, causal=causal)
        o2, lse2 = oracle.attention(q, k + c, v, softmax_scale=scale, causal=causal)
        shift = scale * np.einsum("bihd,d->bhi", q, c)
        assert np.allclose(o2, o, atol=1e-13)
        assert np.allclose(lse2, lse + shift, atol=1e-13)


def test_split_merge_identity():
    rng = np.random.default_rng(9)
    q, k, v = _rand((1, 4, 2, 8), rng), _rand((1, 23, 2, 8), rng), _rand((1, 23, 2, 8), rng)
    o, lse = oracle.attention(q, k, v, softmax_scale=0.5)
    cuts = [0, 5, 6, 17, 23]
    parts = [oracle.attention(q, k[:, a:b], v[:, a:b], softmax_scale=0.5)
             for a, b in zip(cuts[:-1], cuts[1:])]
    om, lm = oracle.merge_partials([p[0] for p in parts],
                                   [np.transpose(p[1], (0, 2, 1))[..., None].squeeze(-1)
                                    for p in parts])
    assert np.allclose(om, o, atol=1e-13)
    assert np.allclose(lm, np.transpose(lse, (0, 2, 1)), atol=1e-13)


def test_merge_with_empty_chunk():
    o1 = np.array([[1.0, 2.0]])
    l1 = np.array([0.5])
    oe = np.zeros((1, 2))
    le = np.array([-np.inf])
    om, lm = oracle.merge_partials([o1, oe], [l1, le])
    assert np.allclose(om, o1) and np.allclose(lm, l1)
    om, lm = oracle.merge_partials([oe, oe], [le, le])
    assert np.all(om == 0) and np.all(lm == -np.inf)


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_fp64(causal):
    """Library cross-check: torch's fp64 CPU attention (top-left causal == ours when Sq == Sk)."""
    rng = np.random.default_rng(10)
    B, S, H, D = 2, 33, 3, 16
    q, k, v = (torch.from_numpy(_rand((B, S, H, D), rng)) for _ in range(3))
    scale = D ** -0.5
    o, lse = oracle.attention(q, k, v, softmax_scale=scale, causal=causal)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q.transpose(1, 2), k.transpose(1, 2), v.transpose(1, 2), is_causal=causal,
        scale=scale).transpose(1, 2)
    assert np.allclose(o, ref.numpy(), atol=1e-13)
    s = torch.einsum("bihd,bjhd->bhij", q, k) * scale
    if causal:
        s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), -math.inf)
    assert np.allclose(lse, torch.logsumexp(s, dim=-1).numpy(), atol=1e-13)


def test_varlen_equals_per_sequence():
    rng = np.random.default_rng(11)
    sq = [3, 0, 5, 2]
    sk = [4, 2, 5, 0]
    H, D = 2, 4
    cq = np.concatenate([[0], np.cumsum(sq)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(sk)]).astype(np.int32)
    q, k, v = _rand((cq[-1], H, D), rng), _rand((ck[-1], H, D), rng), _rand((ck[-1], H, D), rng)
    for causal in (False, True):
        o, lse = oracle.attention(q, k, v, softmax_scale=0.5, causal=causal,
                                  cu_seqlens_q=cq, cu_seqlens_k=ck)
        for b in range(4):
            if sq[b] == 0:
                continue
            qb = q[cq[b]:cq[b + 1]][None]
            kb = k[ck[b]:ck[b + 1]][None]
            vb = v[ck[b]:ck[b + 1]][None]
            ob, lb = oracle.attention(qb, kb, vb, softmax_scale=0.5, causal=causal)
            assert np.allclose(o[cq[b]:cq[b + 1]], ob[0], atol=1e-14)
            assert np.array_equal(lse[:, cq[b]:cq[b + 1]], lb[0])


def test_bf16_decoder_matches_torch():
    rng = np.random.default_rng(12)
    codes = rng.integers(0, 1 << 16, size=20000, dtype=np.uint16)
    vals = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.decode(codes, oracle.DT_BF16)
    finite = np.isfinite(vals)
    assert np.array_equal(got[finite], vals[finite])
    assert np.array_equal(np.isnan(got), np.isnan(vals))


def test_e4m3_decoder_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.decode(codes, oracle.DT_E4M3)
    nan = np.isnan(vals)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(got[~nan], vals[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_fp8_descale_equals_dequantised_fp64():
    from exact_attention_forward_gb300 import inputs
    g = torch.Generator().manual_seed(13)
    x = [torch.randn((1, 16, 2, 8), generator=g) for _ in range(3)]
    qs = [inputs.quantize_e4m3(t) for t in x]
    (q8, dq), (k8, dk), (v8, dv) = qs
    o, lse = oracle.attention(q8, k8, v8, softmax_scale=0.3, descale=(dq, dk, dv))
    deq = [t.to(torch.float64) * d for t, d in qs]
    o2, lse2 = oracle.attention(*deq, softmax_scale=0.3)
    assert np.allclose(o, o2, atol=1e-13) and np.allclose(lse, lse2, atol=1e-13)
    # and descale really enters: q_descale scales the scores, v_descale the output
    o3, _ = oracle.attention(q8, k8, v8, softmax_scale=0.3, descale=(dq, dk, 2 * dv))
    assert np.allclose(o3, 2 * o, atol=1e-13)


def test_rows_subset_equals_full():
    rng = np.random.default_rng(14)
    q, k, v = _rand((2, 10, 3, 4), rng), _rand((2, 10, 3, 4), rng), _rand((2, 10, 3, 4), rng)
    o, lse = oracle.attention(q, k, v, softmax_scale=0.5, causal=True)
    rows = np.array([[1, 2, 9], [0, 0, 0], [1, 0, 4]])
    o_r, l_r = oracle.attention_rows(q, k, v, rows, softmax_scale=0.5, causal=True)
    for r, (b, h, i) in enumerate(rows):
        assert np.array_equal(o_r[r], o[b, i, h]) and l_r[r] == lse[b, h, i]


def test_bad_arguments_rejected():
    q = np.zeros((1, 2, 1, 4))
    with pytest.raises(ValueError):
        oracle.attention_rows(q, q, q, np.array([[0, 0, 5]]), softmax_scale=1.0)
    with pytest.raises(ValueError):
        oracle.attention_rows(q, q, q, np.array([[0, 3, 0]]), softmax_scale=1.0)


def test_huge_scores_stay_finite_and_match_closed_form():
    """Scores in the thousands: exp overflows unless the true row max is subtracted.
    Keys k_j = (j, 1, 0...) and q = (40, 0, ...) give s_j = 40 j * scale; the softmax
    weights are w_j = exp(s_j - s_max) / sum, the LSE is s_max + ln sum_j exp(s_j - s_max)."""
    n, d, scale = 9, 4, 7.0
    q = np.zeros((1, 1, 1, d))
    q[0, 0, 0, 0] = 40.0
    k = np.zeros((1, n, 1, d))
    k[0, :, 0, 0] = np.arange(n)
    k[0, :, 0, 1] = 1.0
    v = np.zeros((1, n, 1, 2))
    v[0, :, 0, 0] = np.arange(n) * 1.5 - 3.0
    v[0, :, 0, 1] = 1.0
    s = [40.0 * j * scale for j in range(n)]   # up to 2240
    smax = max(s)
    z = sum(math.exp(x - smax) for x in s)
    o, lse = oracle.attention(q, k, v, softmax_scale=scale)
    assert np.all(np.isfinite(o)) and np.isfinite(lse).all()
    assert lse[0, 0, 0] == pytest.approx(smax + math.log(z), rel=1e-14)
    expect0 = sum(math.exp(x - smax) * (j * 1.5 - 3.0) for j, x in enumerate(s)) / z
    assert o[0, 0, 0, 0] == pytest.approx(expect0, abs=1e-12)
    assert o[0, 0, 0, 1] == pytest.approx(1.0, abs=1e-14)
    # causal, Sq = Sk: row i sees keys 0..i, so the newest key dominates every row
    qq = np.repeat(q, n, axis=1)
    o2, lse2 = oracle.attention(qq, k, v, softmax_scale=scale, causal=True)
    assert np.all(np.isfinite(o2)) and np.all(np.isfinite(lse2))
    for i in range(n):
        zi = sum(math.exp(s[j] - s[i]) for j in range(i + 1))
        assert lse2[0, 0, i] == pytest.approx(s[i] + math.log(zi), rel=1e-14)


@pytest.mark.parametrize("H,Hk", [(8, 2), (6, 1), (4, 4)])
def test_grouped_query_equals_repeated_heads(H, Hk):
    """Grouped-query attention is multi-head attention over K/V heads repeated so that
    consecutive query heads share one key/value head."""
    rng = np.random.default_rng(15 + H + Hk)
    B, Sq, Sk, D = 2, 7, 11, 5
    q, k, v = _rand((B, Sq, H, D), rng), _rand((B, Sk, Hk, D), rng), _rand((B, Sk, Hk, D), rng)
    kr, vr = np.repeat(k, H // Hk, axis=2), np.repeat(v, H // Hk, axis=2)
    for causal in (False, True):
        o, lse = oracle.attention(q, k, v, softmax_scale=0.4, causal=causal)
        o2, lse2 = oracle.attention(q, kr, vr, softmax_scale=0.4, causal=causal)
        assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_grouped_query_rejects_indivisible_heads():
    q = np.zeros((1, 2, 3, 4))
    k = np.zeros((1, 2, 2, 4))
    with pytest.raises(ValueError):
        oracle.attention(q, k, k, softmax_scale=1.0)


# --------------------------------------------------------------------------
# FP8 with per-(batch, head) descales and an E5M2 V; per-sequence key
# lengths inside a fixed-capacity cache; appending new keys to that cache
# --------------------------------------------------------------------------
def test_e5m2_decoder_matches_fp16_bits_and_torch():
    codes = np.arange(256, dtype=np.uint8)
    # an E5M2 code is the high byte of an IEEE binary16 of the same value
    half = (codes.astype(np.uint16) << 8).view(np.float16).astype(np.float64)
    tvals = torch.from_numpy(codes).view(torch.float8_e5m2).to(torch.float64).numpy()
    got = oracle.decode(codes, oracle.DT_E5M2)
    nan = np.isnan(half)
    assert np.array_equal(nan, np.isnan(got)) and np.array_equal(nan, np.isnan(tvals))
    assert np.array_equal(got[~nan], half[~nan]) and np.array_equal(got[~nan], tvals[~nan])
    assert got[0x7B] == 57344.0 and got[0x01] == 2.0 ** -16 and got[0x7C] == np.inf
    assert got[0xFC] == -np.inf and got[0x04] == 2.0 ** -14


@pytest.mark.parametrize("H, Hk, causal", [(4, 4, False), (4, 2, True), (3, 1, True)])
def test_per_head_descale_equals_dequantised_fp64(H, Hk, causal):
    from exact_attention_forward_gb300 import inputs
    g = torch.Generator().manual_seed(40 + H + Hk)
    B, Sq, Sk, D = 3, 9, 13, 8
    # per-head amplitudes differ so that a descale read from the wrong (b, head) shows
    amp_q = torch.rand((B, 1, H, 1), generator=g) * 3 + 0.2
    amp_k = torch.rand((B, 1, Hk, 1), generator=g) * 3 + 0.2
    q = torch.randn((B, Sq, H, D), generator=g) * amp_q
    k = torch.randn((B, Sk, Hk, D), generator=g) * amp_k
    v = torch.randn((B, Sk, Hk, D), generator=g) * amp_k
    q8, dq = inputs.quantize_fp8_per_head(q, "e4m3", Hk)
    k8, dk = inputs.quantize_fp8_per_head(k, "e4m3", Hk)
    v8, dv = inputs.quantize_fp8_per_head(v, "e5m2", Hk)
    assert q8.dtype == torch.float8_e4m3fn and v8.dtype == torch.float8_e5m2
    o, lse = oracle.attention(q8, k8, v8, softmax_scale=0.3, causal=causal, descale=(dq, dk, dv))
    # dequantise with torch's own FP8 decoders: each (b, head) slice times its descale
    grp = H // Hk
    d64 = lambda t: t.to(torch.float64)
    deq_q = d64(q8) * d64(dq).repeat_interleave(grp, dim=1)[:, None, :, None]
    deq_k = d64(k8) * d64(dk)[:, None, :, None]
    deq_v = d64(v8) * d64(dv)[:, None, :, None]
    o2, lse2 = oracle.attention(deq_q, deq_k, deq_v, softmax_scale=0.3, causal=causal)
    assert np.allclose(o, o2, rtol=0, atol=1e-12) and np.allclose(lse, lse2, rtol=0, atol=1e-12)
    O, L = brute_force(deq_q.numpy().tolist(), deq_k.numpy().tolist(), deq_v.numpy().tolist(),
                       0.3, causal)
    assert np.allclose(o, np.array(O), rtol=0, atol=1e-10)
    assert np.allclose(lse, np.array(L), rtol=0, atol=1e-10)
    # a scalar descale is the same as a constant per-head array
    o3, lse3 = oracle.attention(q8, k8, v8, softmax_scale=0.3, causal=causal,
                                descale=(0.5, 0.25, 2.0))
    o4, lse4 = oracle.attention(q8, k8, v8, softmax_scale=0.3, causal=causal,
                                descale=(np.full((B, Hk), 0.5), np.full((B, Hk), 0.25),
                                         np.full((B, Hk), 2.0)))
    assert np.array_equal(o3, o4) and np.array_equal(lse3, lse4)


@pytest.mark.parametrize("causal", [False, True])
def test_seqused_k_equals_truncated_keys(causal):
    rng = np.random.default_rng(41)
    B, Sq, cap, H, Hk, D = 4, 5, 11, 2, 1, 4
    used = [11, 0, 6, 3]          # full, empty, partial, shorter than Sq
    q, k, v = _rand((B, Sq, H, D), rng), _rand((B, cap, Hk, D), rng), _rand((B, cap, Hk, D), rng)
    o, lse = oracle.attention(q, k, v, softmax_scale=0.7, causal=causal, seqused_k=used)
    for b in range(B):
        u = used[b]
        if u == 0:
            assert np.all(o[b] == 0) and np.all(lse[b] == -np.inf)
            continue
        O, L = brute_force(q[b:b + 1].tolist(), k[b:b + 1, :u].tolist(), v[b:b + 1, :u].tolist(),
                           0.7, causal)
        L = np.array(L)[0]
        fin = np.isfinite(L)
        assert np.array_equal(fin, np.isfinite(lse[b]))
        assert np.allclose(lse[b][fin], L[fin], rtol=0, atol=1e-12)
        O = np.array([[row if row is not None else [0.0] * D for row in r] for r in O[0]])
        assert np.allclose(o[b], O, rtol=0, atol=1e-12)
    with pytest.raises(ValueError):  # more keys used than stored
        oracle.attention(q, k, v, softmax_scale=0.7, seqused_k=[12, 0, 0, 0])


def test_append_kv_writes_rows_and_attention_sees_them():
    g = torch.Generator().manual_seed(42)
    B, cap, Hk, H, D, n_new = 3, 12, 2, 4, 8, 4
    seqlens = [3, 0, 8]
    cache = torch.randn((B, cap, Hk, D), generator=g).to(torch.bfloat16)
    new = torch.randn((B, n_new, Hk, D), generator=g).to(torch.bfloat16)
    before = cache.clone()
    out = oracle.append_kv(cache, new, seqlens)
    assert out.dtype == torch.bfloat16 and torch.equal(cache, before)  # input untouched
    for b, s in enumerate(seqlens):
        assert torch.equal(out[b, :s], cache[b, :s])
        assert torch.equal(out[b, s:s + n_new], new[b])
        assert torch.equal(out[b, s + n_new:], cache[b, s + n_new:])
    with pytest.raises(ValueError):
        oracle.append_kv(cache, new, [3, 0, 9])  # 9 + 4 > capacity
    # attention of the new queries over the grown cache == torch SDPA (fp64, explicit
    # bottom-right causal mask) over the concatenation of old prefix and new keys
    vcache = torch.randn((B, cap, Hk, D), generator=g).to(torch.bfloat16)
    vnew = torch.randn((B, n_new, Hk, D), generator=g).to(torch.bfloat16)
    kc, vc = out, oracle.append_kv(vcache, vnew, seqlens)
    q = torch.randn((B, n_new, H, D), generator=g).to(torch.bfloat16)
    used = [s + n_new for s in seqlens]
    o, lse = oracle.attention(q, kc, vc, softmax_scale=0.35, causal=True, seqused_k=used)
    for b, s in enumerate(seqlens):
        kk = torch.cat([cache[b, :s], new[b]]).to(torch.float64).repeat_interleave(H // Hk, dim=1)
        vv = torch.cat([vcache[b, :s], vnew[b]]).to(torch.float64).repeat_interleave(H // Hk, dim=1)
        qq = q[b].to(torch.float64)
        sk = s + n_new
        mask = torch.arange(sk)[None, :] <= torch.arange(n_new)[:, None] + (sk - n_new)
        ref = torch.nn.functional.scaled_dot_product_attention(
            qq.transpose(0, 1), kk.transpose(0, 1), vv.transpose(0, 1), attn_mask=mask, scale=0.35)
        assert np.allclose(o[b], ref.transpose(0, 1).numpy(), rtol=0, atol=1e-12)
