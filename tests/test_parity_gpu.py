"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs, element by element.

Every comparison covers every row.  Small shapes span several tiles plus
ragged tails in both the query and key directions; the configured workloads
(up to 2 x 32 x 8192 query rows) run at full size in the launch configuration
the benchmark times.  Outputs start as NaN, so a row the schedule never wrote
fails the comparison.
"""
import numpy as np
import pytest
import torch

import oracle
import exact_attention_forward_gb300 as fa
from exact_attention_forward_gb300 import inputs
from parity_util import compare, oracle_abs_v, nan_outputs, oracle_full, run_gpu, to_dev, workload_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    fa.debug_set(0, 0)
    fa.device_error(clear=True)


SMALL = [
    # B, H, Sq, Sk, D, causal
    (1, 1, 128, 128, 128, False),
    (1, 1, 128, 128, 128, True),
    (2, 3, 1, 1, 64, False),
    (1, 2, 127, 129, 128, False),
    (1, 2, 129, 127, 128, True),
    (2, 2, 255, 300, 64, True),
    (1, 1, 513, 257, 128, False),
    (1, 2, 300, 513, 128, True),   # Sq < Sk: bottom-right diagonal
    (1, 2, 513, 300, 128, True),   # Sq > Sk: leading rows see no key
    (1, 1, 3, 1000, 128, False),
    (1, 4, 384, 384, 64, True),
    (3, 2, 640, 640, 128, True),
    (1, 1, 1024, 1024, 128, False),
]


@pytest.mark.parametrize("B,H,Sq,Sk,D,causal", SMALL)
def test_small_shapes_full(B, H, Sq, Sk, D, causal):
    x = inputs.make_random(B, H, Sq, Sk, D, seed=17 + Sq + 3 * Sk + D)
    scale = D ** -0.5
    o, lse = run_gpu(x, causal=causal, softmax_scale=scale)
    o_ref, lse_ref = oracle.attention(x["q"], x["k"], x["v"], softmax_scale=scale, causal=causal)
    compare(o, lse, o_ref, lse_ref, what=f"{(B, H, Sq, Sk, D, causal)}")


@pytest.mark.parametrize("name", ["bf16_small", "bf16_causal_2k"])
def test_small_and_2k_workloads_full(name):
    w = inputs.WORKLOADS[name]
    x = workload_inputs(name)
    o, lse = run_gpu(x, causal=w.causal, softmax_scale=w.softmax_scale)
    o_ref, lse_ref = oracle_full(name)
    compare(o, lse, o_ref, lse_ref, what=w.name)


@pytest.mark.parametrize("name", ["bf16_causal_8k", "bf16_noncausal_8k"])
def test_8k_workloads_full(name):
    # every row of the 2 x 32 x 8192 query rows against the fp64 oracle, in the launch
    # configuration the benchmark times (L2 bands, LPT snake, single-tile tail)
    w = inputs.WORKLOADS[name]
    x = workload_inputs("bf16_causal_8k")  # both workloads attend over the same inputs
    o, lse = run_gpu(x, causal=w.causal, softmax_scale=w.softmax_scale)
    o_ref, lse_ref = oracle_full(name)
    compare(o, lse, o_ref, lse_ref, what=name,
            o_abs_v=oracle_abs_v(x, softmax_scale=w.softmax_scale, causal=w.causal))


def test_varlen_workload_full():
    w = inputs.WORKLOADS["bf16_varlen_causal"]
    x = workload_inputs(w.name)
    sq, sk = x["seqlens"]
    cu_q = x["cu_seqlens_q"].numpy()
    o, lse = run_gpu(x, causal=w.causal, softmax_scale=w.softmax_scale)
    o_ref, lse_ref = oracle_full(w.name)
    compare(o, lse, o_ref, lse_ref, what=w.name)
    # the sequences without keys: every row exactly O = 0, LSE = -inf
    for b in w.empty_k_at:
        assert sk[b] == 0 and sq[b] > 0
        sl = slice(cu_q[b], cu_q[b + 1])
        assert np.all(o[sl] == 0) and np.all(lse[:, sl] == -np.inf)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_small_full(causal):
    sq = [5, 0, 130, 257, 1, 128, 40]
    sk = [7, 3, 0, 300, 1, 128, 40]
    x = inputs.make_varlen(sq, sk, heads=3, head_dim=128, seed=21)
    o, lse = run_gpu(x, causal=causal, softmax_scale=128 ** -0.5)
    o_ref, lse_ref = oracle.attention(x["q"], x["k"], x["v"], softmax_scale=128 ** -0.5,
                                      causal=causal, cu_seqlens_q=x["cu_seqlens_q"],
                                      cu_seqlens_k=x["cu_seqlens_k"])
    compare(o, lse, o_ref, lse_ref, what=f"varlen small causal={causal}")


def test_fp8_small_full():
    w = inputs.Workload("fp8_small", 2, 3, 300, 400, 128, False, dtype="e4m3", seed=31)
    x = inputs.make_inputs(w)
    for causal in (False, True):
        o, lse = run_gpu(x, causal=causal, softmax_scale=w.softmax_scale)
        o_ref, lse_ref = oracle.attention(x["q"], x["k"], x["v"], softmax_scale=w.softmax_scale,
                                          causal=causal, descale=x["descale"])
        compare(o, lse, o_ref, lse_ref, dtype="e4m3", what=f"fp8 small causal={causal}")


def test_fp8_workload_full():
    w = inputs.WORKLOADS["fp8_noncausal_4k"]
    x = workload_inputs(w.name)
    o, lse = run_gpu(x, causal=w.causal, softmax_scale=w.softmax_scale)
    o_ref, lse_ref = oracle_full(w.name)
    compare(o, lse, o_ref, lse_ref, dtype="e4m3", what=w.name)


def test_shortq_longkv_split_and_unsplit():
    w = inputs.WORKLOADS["bf16_shortq_longkv"]
    x = workload_inputs(w.name)
    assert fa.num_splits(w.batch, w.heads, w.seqlen_q, w.seqlen_k) > 1
    o_s, lse_s = run_gpu(x, causal=False, softmax_scale=w.softmax_scale, workspace="auto")
    o_n, lse_n = run_gpu(x, causal=False, softmax_scale=w.softmax_scale, workspace=None)
    o_ref, lse_ref = oracle_full(w.name)
    compare(o_s, lse_s, o_ref, lse_ref, what=w.name)
    compare(o_n, lse_n, o_ref, lse_ref, what="short-q long-kv, unsplit")


@pytest.mark.parametrize("D,causal", [(128, False), (128, True), (64, False)])
def test_varlen_split(D, causal):
    # a packed batch of short query blocks against long (and empty) key ranges: the key
    # range is split over CTAs as for fixed-length shapes, with the partial rows laid out
    # per sequence (max_seqlen_q rows each) and merged into the packed outputs
    sq = [1, 37, 0, 128, 5]
    sk = [20000, 5000, 3000, 30000, 0]
    x = inputs.make_varlen(sq, sk, heads=4, head_dim=D, seed=61 + D)
    assert fa.num_splits(len(sq), 4, max(sq), max(sk), causal) > 1
    o_s, lse_s = run_gpu(x, causal=causal, softmax_scale=D ** -0.5, workspace="auto")
    o_n, lse_n = run_gpu(x, causal=causal, softmax_scale=D ** -0.5, workspace=None)
    o_ref, lse_ref = oracle.attention(x["q"], x["k"], x["v"], softmax_scale=D ** -0.5,
                                      causal=causal, cu_seqlens_q=x["cu_seqlens_q"],
                                      cu_seqlens_k=x["cu_seqlens_k"])
    compare(o_s, lse_s, o_ref, lse_ref, what=f"varlen split D={D} causal={causal}")
    compare(o_n, lse_n, o_ref, lse_ref, what=f"varlen unsplit D={D} causal={causal}")


def test_split_causal_small():
    # causal with a short query block against a long key range: splits whose
    # key range lies beyond every row's diagonal produce -inf partials
    x = inputs.make_random(1, 2, 200, 6000, 128, seed=41)
    assert fa.num_splits(1, 2, 200, 6000, causal=True) > 1
    o, lse = run_gpu(x, causal=True, softmax_scale=128 ** -0.5)
    o_ref, lse_ref = oracle.attention(x["q"], x["k"], x["v"], softmax_scale=128 ** -0.5,
                                      causal=True)
    compare(o, lse, o_ref, lse_ref, what="split causal")


@pytest.mark.parametrize("D", [128, 64])
def test_many_splits(D):
    # one (batch, head) and a long key range: more than 32 key splits, so the merge's
    # per-split weights no longer fit one per lane
    x = inputs.make_random(1, 1, 100, 40000, D, seed=43 + D)
    assert fa.num_splits(1, 1, 100, 40000) > 32
    o, lse = run_gpu(x, causal=False, softmax_scale=D ** -0.5)
    o_ref, lse_ref = oracle.attention(x["q"], x["k"], x["v"], softmax_scale=D ** -0.5)
    compare(o, lse, o_ref, lse_ref, what=f"many splits D={D}")


@pytest.mark.parametrize("B,H,Hk,Sq,Sk,D,causal", [
    (2, 8, 2, 300, 513, 128, False),
    (2, 8, 2, 513, 513, 128, True),
    (1, 6, 3, 257, 130, 64, True),
    (1, 16, 1, 128, 3000, 128, False),   # multi-query; splits the key range
])
def test_grouped_query_full(B, H, Hk, Sq, Sk, D, causal):
    x = inputs.make_random(B, H, Sq, Sk, D, seed=90 + H + Hk + Sq, heads_k=Hk)
    o, lse = run_gpu(x, causal=causal, softmax_scale=D ** -0.5)
    o_ref, lse_ref = oracle.attention(x["q"], x["k"], x["v"], softmax_scale=D ** -0.5,
                                      causal=causal)
    compare(o, lse, o_ref, lse_ref, what=f"gqa {(B, H, Hk, Sq, Sk, D, causal)}")


@pytest.mark.parametrize("B,H,Hk,Sq,Sk,D,causal", [
    (2, 8, 2, 64, 700, 128, True),       # group 4 x 64 rows: one full tile pair
    (1, 32, 4, 7, 1000, 128, True),      # group 8 x 7 rows: part of tile 0
    (3, 6, 3, 100, 300, 128, True),      # group 2 x 100 rows: tile 1 partly filled
    (1, 16, 1, 16, 5000, 128, False),    # multi-query, 16 heads x 16 rows, key splits
    (2, 8, 2, 32, 500, 64, True),        # D = 64
    (1, 6, 2, 10, 300, 128, True),       # group 3 does not divide 128: not packed
    (2, 4, 2, 1, 2000, 128, True),       # decoding: one query row
])
def test_grouped_query_packed_tiles(B, H, Hk, Sq, Sk, D, causal):
    # short query blocks: the query heads of a K/V head share the rows of one tile
    x = inputs.make_random(B, H, Sq, Sk, D, seed=120 + H + Hk + Sq + D, heads_k=Hk)
    o, lse = run_gpu(x, causal=causal, softmax_scale=D ** -0.5)
    o_ref, lse_ref = oracle.attention(x["q"], x["k"], x["v"], softmax_scale=D ** -0.5,
                                      causal=causal)
    compare(o, lse, o_ref, lse_ref, what=f"packed gqa {(B, H, Hk, Sq, Sk, D, causal)}")


def test_grouped_query_varlen_and_fp8():
    x = inputs.make_varlen([40, 300, 0, 129], [40, 300, 5, 200], heads=4, head_dim=128, seed=95,
                           heads_k=2)
    o, lse = run_gpu(x, causal=True, softmax_scale=128 ** -0.5)
    o_ref, lse_ref = oracle.attention(x["q"], x["k"], x["v"], softmax_scale=128 ** -0.5,
                                      causal=True, cu_seqlens_q=x["cu_seqlens_q"],
                                      cu_seqlens_k=x["cu_seqlens_k"])
    compare(o, lse, o_ref, lse_ref, what="gqa varlen")
    w = inputs.Workload("fp8_gqa", 2, 4, 200, 300, 128, False, dtype="e4m3", seed=96, heads_k=1)
    x = inputs.make_inputs(w)
    o, lse = run_gpu(x, causal=False, softmax_scale=w.softmax_scale)
    o_ref, lse_ref = oracle.attention(x["q"], x["k"], x["v"], softmax_scale=w.softmax_scale,
                                      descale=x["descale"])
    compare(o, lse, o_ref, lse_ref, dtype="e4m3", what="gqa fp8")


def test_zero_keys_fixed_length():
    x = inputs.make_random(2, 2, 130, 0, 128, seed=3)
    o, lse = run_gpu(x, causal=False, softmax_scale=0.1)
    assert np.all(o == 0) and np.all(lse == -np.inf)


def test_guard_bands_untouched():
    B, H, S, D = 1, 2, 200, 128
    x = to_dev(inputs.make_random(B, H, S, S, D, seed=8))
    pad = 4096
    o_buf = torch.full((2 * pad + B * S * H * D,), 7.0, dtype=torch.bfloat16, device="cuda")
    l_buf = torch.full((2 * pad + B * H * S,), 9.0, dtype=torch.float32, device="cuda")
    o = o_buf[pad:pad + B * S * H * D].view(B, S, H, D)
    lse = l_buf[pad:pad + B * H * S].view(B, H, S)
    fa.fwd(x["q"], x["k"], x["v"], causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(o_buf[:pad] == 7.0) and torch.all(o_buf[-pad:] == 7.0)
    assert torch.all(l_buf[:pad] == 9.0) and torch.all(l_buf[-pad:] == 9.0)
    assert torch.all(torch.isfinite(o))


def test_rejected_call_writes_nothing():
    x = to_dev(inputs.make_random(1, 1, 64, 64, 128, seed=9))
    o = torch.full((1, 64, 1, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((1, 1, 64), 5.0, dtype=torch.float32, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fwd(x["q"], x["k"], x["v"], softmax_scale=-1.0, out=o, lse=lse)
    assert e.value.status == fa.FA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(o == 3.0) and torch.all(lse == 5.0)


def test_deterministic():
    x = to_dev(inputs.make_random(2, 4, 700, 900, 128, seed=10))
    a = nan_outputs(x["q"], x["v"], (2, 4, 700))
    b = nan_outputs(x["q"], x["v"], (2, 4, 700))
    fa.fwd(x["q"], x["k"], x["v"], causal=True, out=a[0], lse=a[1])
    fa.fwd(x["q"], x["k"], x["v"], causal=True, out=b[0], lse=b[1])
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_bounded_wait_timeout_is_reported_and_context_survives():
    x = to_dev(inputs.make_random(1, 2, 256, 256, 128, seed=11))
    fa.device_error(clear=True)
    fa.debug_set(wait_limit_ns=200_000_000, inject=1)  # withhold one Q-tile arrival
    try:
        fa.fwd(x["q"], x["k"], x["v"])
        st, flags = fa.device_error(clear=True)
    finally:
        fa.debug_set(0, 0)
    assert st == fa.FA_ERR_DEVICE_TIMEOUT
    # the first wait to give up is one that depends on the withheld Q arrival: the MMA
    # issuer's Q wait (3), the softmax's S wait (7), or, later in the chain, a K/V ring
    # wait (2, 4) -- which one wins the race to the limit is not fixed
    assert flags & 1 and (flags >> 8) & 0xFF in (2, 3, 4, 7)
    # the context is still usable and results are right again
    o, lse = nan_outputs(x["q"], x["v"], (1, 2, 256))
    fa.fwd(x["q"], x["k"], x["v"], out=o, lse=lse)
    torch.cuda.synchronize()
    assert fa.device_error(clear=True)[0] == fa.FA_OK
    o_ref, lse_ref = oracle.attention(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(),
                                      softmax_scale=128 ** -0.5)
    compare(o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
            o_ref, lse_ref, what="after timeout")
