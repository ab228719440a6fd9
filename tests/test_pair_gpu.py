"""GPU parity of the CTA-pair kernel (fa_fwd_2cta: cta_group::2 MMAs over 256-row
slots, each CTA of a cluster loading half of every K/V block) against the fp64
oracle, on the shapes that exercise what differs from the one-CTA kernel: work
items of 512 query rows whose second CTA's rows run past the sequence end, key
blocks that one CTA of a slot sees fully masked under a causal mask, grouped
K/V heads, varlen batches with empty sequences, and the full-size workloads (every row).
"""
import numpy as np
import pytest
import torch

import oracle
import exact_attention_forward_gb300 as fa
from exact_attention_forward_gb300 import inputs
from parity_util import compare, oracle_abs_v, oracle_full, run_gpu, workload_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    fa.debug_set(0, 0)
    fa.device_error(clear=True)


SHAPES = [
    # B, H, Hk, Sq, Sk, causal
    (1, 1, 1, 128, 128, False),
    (1, 1, 1, 128, 128, True),
    (1, 2, 2, 129, 127, True),
    (1, 2, 2, 300, 513, True),    # Sq < Sk: bottom-right diagonal
    (1, 2, 2, 513, 300, True),    # Sq > Sk: leading rows see no key
    (1, 1, 1, 3, 1000, False),
    (1, 2, 2, 600, 600, True),    # last item: the odd CTA's rows of slot 0 all past the end
    (1, 2, 2, 600, 600, False),
    (1, 1, 1, 700, 700, True),    # last item: slot 1 empty
    (3, 2, 2, 640, 640, True),
    (2, 2, 2, 1100, 1100, True),
    (1, 1, 1, 1024, 1024, False),
    (2, 8, 2, 513, 513, True),    # grouped K/V heads
    (1, 16, 1, 300, 2000, False),  # multi-query
]


@pytest.mark.parametrize("B,H,Hk,Sq,Sk,causal", SHAPES)
def test_pair_small_full(B, H, Hk, Sq, Sk, causal):
    x = inputs.make_random(B, H, Sq, Sk, 128, seed=300 + Sq + 3 * Sk + H, heads_k=Hk)
    scale = 128 ** -0.5
    o, lse = run_gpu(x, causal=causal, softmax_scale=scale, cta_pair=True)
    o_ref, lse_ref = oracle.attention(x["q"], x["k"], x["v"], softmax_scale=scale, causal=causal)
    compare(o, lse, o_ref, lse_ref, what=f"pair {(B, H, Hk, Sq, Sk, causal)}")


def test_pair_no_keys():
    x = inputs.make_random(2, 2, 300, 0, 128, seed=331)
    o, lse = run_gpu(x, causal=False, softmax_scale=128 ** -0.5, cta_pair=True)
    assert np.all(o == 0) and np.all(lse == -np.inf)


@pytest.mark.parametrize("causal", [False, True])
def test_pair_varlen_small_full(causal):
    sq = [5, 0, 130, 700, 1, 128, 40, 513]
    sk = [7, 3, 0, 650, 1, 128, 40, 900]
    x = inputs.make_varlen(sq, sk, heads=3, head_dim=128, seed=333)
    o, lse = run_gpu(x, causal=causal, softmax_scale=128 ** -0.5, cta_pair=True)
    o_ref, lse_ref = oracle.attention(x["q"], x["k"], x["v"], softmax_scale=128 ** -0.5,
                                      causal=causal, cu_seqlens_q=x["cu_seqlens_q"],
                                      cu_seqlens_k=x["cu_seqlens_k"])
    compare(o, lse, o_ref, lse_ref, what=f"pair varlen causal={causal}")


@pytest.mark.parametrize("name", ["bf16_causal_8k", "bf16_noncausal_8k"])
def test_pair_8k_workloads_full(name):
    w = inputs.WORKLOADS[name]
    x = workload_inputs("bf16_causal_8k")  # both workloads attend over the same inputs
    o, lse = run_gpu(x, causal=w.causal, softmax_scale=w.softmax_scale, cta_pair=True)
    o_ref, lse_ref = oracle_full(name)
    compare(o, lse, o_ref, lse_ref, what=f"pair {name}",
            o_abs_v=oracle_abs_v(x, softmax_scale=w.softmax_scale, causal=w.causal))


def test_pair_varlen_workload_full():
    w = inputs.WORKLOADS["bf16_varlen_causal"]
    x = workload_inputs(w.name)
    o, lse = run_gpu(x, causal=w.causal, softmax_scale=w.softmax_scale, cta_pair=True)
    o_ref, lse_ref = oracle_full(w.name)
    compare(o, lse, o_ref, lse_ref, what=f"pair {w.name}")


def test_pair_rejects_unbuilt_configurations():
    q = torch.zeros(1, 128, 2, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(fa.FaError) as ei:
        fa.fwd(q, q, q, cta_pair=True)
    assert ei.value.status == fa.FA_ERR_UNSUPPORTED
    q8 = torch.zeros(1, 128, 2, 128, device="cuda").to(torch.float8_e4m3fn)
    with pytest.raises(ValueError):
        fa.fwd(q8, q8, q8, cta_pair=True)


def test_pair_bounded_wait_timeout_is_reported_and_context_survives():
    # both CTAs of each pair withhold their Q loads: the even CTA's MMA issuer gives up on
    # its Q barrier, every role of both CTAs leaves through a bounded wait, the pair meets
    # at the closing cluster barrier and frees its TMEM together
    x = inputs.make_random(1, 2, 600, 600, 128, seed=341)
    fa.device_error(clear=True)
    fa.debug_set(wait_limit_ns=200_000_000, inject=1)
    try:
        d = {n: x[n].cuda() for n in "qkv"}
        fa.fwd(d["q"], d["k"], d["v"], causal=True, cta_pair=True)
        st, flags = fa.device_error(clear=True)
    finally:
        fa.debug_set(0, 0)
    assert st == fa.FA_ERR_DEVICE_TIMEOUT and flags & 1
    # the context is still usable and the pair kernel's results are right again
    o, lse = run_gpu(x, causal=True, softmax_scale=128 ** -0.5, cta_pair=True)
    o_ref, lse_ref = oracle.attention(x["q"], x["k"], x["v"], softmax_scale=128 ** -0.5, causal=True)
    compare(o, lse, o_ref, lse_ref, what="pair after timeout")
