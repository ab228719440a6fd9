"""GPU: behaviour that depends on how work is handed out and on state kept between
launches -- the greedy varlen scheduler's per-launch device counters (more launches
than counter slots, two streams at once, recovery after an aborted launch), CUDA graph
capture and replay, extreme shapes (a thousand tiny sequences, a 256K key range,
thousands of one-tile problems), and the L2-banded static item orders, each checked
against the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import exact_attention_forward_gb300 as fa
from exact_attention_forward_gb300 import inputs
from parity_util import compare, lse_shape_of, nan_outputs, run_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    fa.debug_set(0, 0)
    fa.device_error(clear=True)


def _np(o, lse):
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def _varlen_case(lens, heads=4, seed=0):
    x = inputs.make_varlen(lens, lens, heads=heads, head_dim=128, seed=seed)
    d = to_dev(x)
    kw = dict(causal=True, cu_seqlens_q=d["cu_seqlens_q"], cu_seqlens_k=d["cu_seqlens_k"],
              max_seqlen_q=x["max_seqlen_q"], max_seqlen_k=x["max_seqlen_k"])
    return x, d, kw


def _varlen_ref(x):
    return oracle.attention(x["q"], x["k"], x["v"], softmax_scale=128 ** -0.5, causal=True,
                            cu_seqlens_q=x["cu_seqlens_q"], cu_seqlens_k=x["cu_seqlens_k"])


def test_varlen_launches_wrap_the_counter_slots():
    # 300 launches > 256 counter slots: every slot is reused after its last CTA returned it
    # to zero; a slot left non-zero would skip items and change the result
    x, d, kw = _varlen_case([700, 33, 1200, 5, 400], seed=501)
    o0, l0 = nan_outputs(d["q"], d["v"], lse_shape_of(x))
    fa.fwd(d["q"], d["k"], d["v"], out=o0, lse=l0, **kw)
    torch.cuda.synchronize()
    compare(*_np(o0, l0), *_varlen_ref(x), what="first varlen launch")
    o0, l0 = o0.clone(), l0.clone()
    for i in range(300):
        o, lse = fa.fwd(d["q"], d["k"], d["v"], **kw)
        if i % 37 == 0 or i == 299:
            torch.cuda.synchronize()
            assert torch.equal(o, o0) and torch.equal(lse, l0), f"launch {i} differs"
    assert fa.device_error(clear=True)[0] == fa.FA_OK


def test_varlen_on_two_streams_at_once():
    xa, da, kwa = _varlen_case([900, 17, 1500, 260], seed=502)
    xb, db, kwb = _varlen_case([64, 2000, 3, 700, 700], heads=6, seed=503)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    oa, la = nan_outputs(da["q"], da["v"], lse_shape_of(xa))
    ob, lb = nan_outputs(db["q"], db["v"], lse_shape_of(xb))
    torch.cuda.synchronize()
    for _ in range(20):
        with torch.cuda.stream(sa):
            fa.fwd(da["q"], da["k"], da["v"], stream=sa, out=oa, lse=la, **kwa)
        with torch.cuda.stream(sb):
            fa.fwd(db["q"], db["k"], db["v"], stream=sb, out=ob, lse=lb, **kwb)
    torch.cuda.synchronize()
    assert fa.device_error(clear=True)[0] == fa.FA_OK
    compare(*_np(oa, la), *_varlen_ref(xa), what="stream a")
    compare(*_np(ob, lb), *_varlen_ref(xb), what="stream b")


def test_counter_slot_recovers_after_an_aborted_launch():
    x, d, kw = _varlen_case([600, 250, 1000], seed=504)
    fa.device_error(clear=True)
    fa.debug_set(wait_limit_ns=200_000_000, inject=1)  # withhold one Q-tile arrival: abort
    try:
        fa.fwd(d["q"], d["k"], d["v"], **kw)
        st, _ = fa.device_error(clear=True)
    finally:
        fa.debug_set(0, 0)
    assert st == fa.FA_ERR_DEVICE_TIMEOUT
    # 260 more launches pass over every counter slot, the aborted launch's included
    ref = _varlen_ref(x)
    first = None
    for i in range(260):
        o, lse = nan_outputs(d["q"], d["v"], lse_shape_of(x))
        fa.fwd(d["q"], d["k"], d["v"], out=o, lse=lse, **kw)
        if first is None:
            torch.cuda.synchronize()
            compare(*_np(o, lse), *ref, what="after the aborted launch")
            first = (o.clone(), lse.clone())
        elif i % 29 == 0 or i == 259:
            torch.cuda.synchronize()
            assert torch.equal(o, first[0]) and torch.equal(lse, first[1]), f"launch {i} differs"
    assert fa.device_error(clear=True)[0] == fa.FA_OK


@pytest.mark.parametrize("varlen", [False, True])
def test_cuda_graph_capture_and_replay(varlen):
    if varlen:
        x, d, kw = _varlen_case([300, 129, 1000], seed=505)
        q, k, v = d["q"], d["k"], d["v"]
    else:
        x = inputs.make_random(2, 4, 600, 900, 128, seed=506)
        d = to_dev(x)
        q, k, v = d["q"], d["k"], d["v"]
        kw = dict(causal=True)
    # eager, same arguments as the captured call (no workspace: a key split would change
    # the summation order); also warms the library's per-device state before capture
    o_e, l_e = fa.fwd(q, k, v, workspace=None, **kw)
    torch.cuda.synchronize()
    out, lse = nan_outputs(q, v, tuple(l_e.shape))
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fa.fwd(q, k, v, out=out, lse=lse, workspace=None, stream=s, **kw)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, o_e) and torch.equal(lse, l_e)
    assert fa.device_error(clear=True)[0] == fa.FA_OK
    ref = _varlen_ref(x) if varlen else oracle.attention(x["q"], x["k"], x["v"],
                                                          softmax_scale=128 ** -0.5, causal=True)
    compare(*_np(out, lse), *ref, what="graph replay")


def test_a_thousand_tiny_sequences():
    rng = np.random.default_rng(507)
    sq = [int(v) for v in rng.integers(0, 21, size=1000)]
    sk = [int(v) if rng.random() > 0.05 else 0 for v in rng.integers(0, 21, size=1000)]
    x = inputs.make_varlen(sq, sk, heads=2, head_dim=64, seed=508)
    o, lse = run_gpu(x, causal=True, softmax_scale=64 ** -0.5)
    o_ref, lse_ref = oracle.attention(x["q"], x["k"], x["v"], softmax_scale=64 ** -0.5,
                                      causal=True, cu_seqlens_q=x["cu_seqlens_q"],
                                      cu_seqlens_k=x["cu_seqlens_k"])
    compare(o, lse, o_ref, lse_ref, what="1000 tiny sequences")


def test_256k_key_range():
    # one (batch, head), 2048 key blocks: the maximum of 152-way key splitting
    x = inputs.make_random(1, 1, 64, 262144, 128, seed=509)
    assert fa.num_splits(1, 1, 64, 262144) > 100
    o, lse = run_gpu(x, causal=False, softmax_scale=128 ** -0.5)
    o_ref, lse_ref = oracle.attention(x["q"], x["k"], x["v"], softmax_scale=128 ** -0.5)
    compare(o, lse, o_ref, lse_ref, what="256K keys")


def test_thousands_of_one_tile_problems():
    x = inputs.make_random(64, 32, 128, 128, 128, seed=511)
    o, lse = run_gpu(x, causal=True, softmax_scale=128 ** -0.5)
    o_ref, lse_ref = oracle.attention(x["q"], x["k"], x["v"], softmax_scale=128 ** -0.5,
                                      causal=True)
    compare(o, lse, o_ref, lse_ref, what="64 x 32 one-tile problems")


# Fixed-length static schedules run in L2 bands (consecutive query-tile pairs of one
# (batch, head) side by side).  On a 152-SM GB300 these shapes take the band layouts
# that the large workloads use, at sizes the oracle checks in full: a causal band of
# 2 levels (152 items per level), a causal band of 4 levels with a partial last round
# and the K/V heads shared by groups of 4 query heads, and head-major orders without a
# causal mask (one CTA per SM, and on CTA pairs).  Whatever the order, every item must
# be computed exactly once.
@pytest.mark.parametrize("shape", [
    dict(batch=2, heads=76, heads_k=76, s=1024, d=64, causal=True, pair=False),
    dict(batch=1, heads=76, heads_k=19, s=1792, d=128, causal=True, pair=False),
    dict(batch=3, heads=20, heads_k=20, s=1536, d=64, causal=False, pair=False),
    dict(batch=3, heads=20, heads_k=5, s=1536, d=128, causal=False, pair=True),
], ids=["causal-2-levels", "causal-4-levels-gqa", "noncausal-head-major",
        "noncausal-head-major-pair"])
def test_l2_band_orders(shape):
    s, d = shape["s"], shape["d"]
    x = inputs.make_random(shape["batch"], shape["heads"], s, s, d, seed=521,
                           heads_k=shape["heads_k"])
    scale = d ** -0.5
    o, lse = run_gpu(x, causal=shape["causal"], softmax_scale=scale, workspace=None,
                     cta_pair=shape["pair"])
    o_ref, lse_ref = oracle.attention(x["q"], x["k"], x["v"], softmax_scale=scale,
                                      causal=shape["causal"])
    compare(o, lse, o_ref, lse_ref, what=f"banded order {shape}")


# Without a causal mask, a static schedule whose last round holds at most half as many
# tile pairs as there are CTAs runs that round's pairs as single tiles (two items each).
# On a 152-SM GB300 these shapes take that path: 160 pairs (a tail of 8), 212 pairs (a
# tail of 60) whose last level's second tile holds 4 rows or lies wholly past the end,
# grouped K/V heads, head dim 64 and FP8.
@pytest.mark.parametrize("shape", [
    dict(heads=40, heads_k=40, s=1000, d=128, dtype="bf16"),
    dict(heads=53, heads_k=53, s=900, d=64, dtype="bf16"),
    dict(heads=52, heads_k=13, s=800, d=128, dtype="bf16"),
    dict(heads=40, heads_k=40, s=1000, d=128, dtype="e4m3"),
], ids=["tail-8", "tail-60-ragged", "tail-gqa-empty-tile", "tail-fp8"])
def test_single_tile_tail(shape):
    s, d = shape["s"], shape["d"]
    x = inputs.make_random(1, shape["heads"], s, s, d, seed=541, heads_k=shape["heads_k"],
                           dtype=shape["dtype"])
    scale = d ** -0.5
    o, lse = run_gpu(x, causal=False, softmax_scale=scale, workspace=None)
    o_ref, lse_ref = oracle.attention(x["q"], x["k"], x["v"], softmax_scale=scale,
                                      descale=x["descale"])
    compare(o, lse, o_ref, lse_ref, dtype=shape["dtype"], what=f"single-tile tail {shape}")
