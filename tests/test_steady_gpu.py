"""GPU: the kernel instances for long bf16 head_dim-128 launches (the MMA issuer runs the
middle key blocks of a work item without per-block tests), fixed-length and packed
varlen.  The library picks them by launch size; here fa_debug_select_steady forces them
onto small shapes -- ragged query and key tails, causal with Sq < Sk and Sq > Sk, items of
one and two key blocks, grouped K/V heads, packed sequences with empty ranges -- compared element by element with the fp64 oracle (outputs
pre-filled with NaN) and byte for byte with the other instance, which issues the same
MMAs in the same order."""
import numpy as np
import pytest

import oracle
import exact_attention_forward_gb300 as fa
from exact_attention_forward_gb300 import inputs
from parity_util import compare, run_gpu, workload_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    fa.debug_set(0, 0)
    fa.device_error(clear=True)
    yield
    fa.debug_select_steady(0)


SHAPES = [
    # B, H, Sq, Sk, causal (D = 128)
    (1, 1, 128, 128, True),      # one key block per tile: no steady block
    (1, 2, 256, 2048, False),    # one tile pair, 16 key blocks
    (1, 2, 256, 2048, True),     # Sq < Sk: bottom-right diagonal, long steady run
    (1, 2, 2048, 256, True),     # Sq > Sk: leading rows see no key
    (2, 3, 700, 1500, True),     # ragged query and key tails
    (1, 2, 129, 1000, False),    # tile 1 holds one row
    (3, 2, 640, 640, True),
    (1, 1, 1024, 1024, False),
]


def _both(x, **kw):
    fa.debug_select_steady(1)
    o1, l1 = run_gpu(x, **kw)
    fa.debug_select_steady(-1)
    o0, l0 = run_gpu(x, **kw)
    fa.debug_select_steady(0)
    st, flags = fa.device_error(clear=True)
    assert st == 0, hex(flags)
    return (o1, l1), (o0, l0)


@pytest.mark.parametrize("B,H,Sq,Sk,causal", SHAPES)
def test_steady_instance_small_shapes(B, H, Sq, Sk, causal):
    D = 128
    x = inputs.make_random(B, H, Sq, Sk, D, seed=71 + Sq + 5 * Sk)
    scale = D ** -0.5
    (o1, l1), (o0, l0) = _both(x, causal=causal, softmax_scale=scale)
    o_ref, lse_ref = oracle.attention(x["q"], x["k"], x["v"], softmax_scale=scale, causal=causal)
    compare(o1, l1, o_ref, lse_ref, what=f"steady instance {(B, H, Sq, Sk, causal)}")
    assert np.array_equal(o1, o0) and np.array_equal(l1, l0)


def test_steady_instance_grouped_heads():
    B, H, Hk, Sq, Sk, D = 2, 8, 2, 600, 1800, 128
    x = inputs.make_random(B, H, Sq, Sk, D, seed=907, heads_k=Hk)
    scale = D ** -0.5
    (o1, l1), (o0, l0) = _both(x, causal=True, softmax_scale=scale)
    o_ref, lse_ref = oracle.attention(x["q"], x["k"], x["v"], softmax_scale=scale, causal=True)
    compare(o1, l1, o_ref, lse_ref, what="steady instance, grouped K/V heads")
    assert np.array_equal(o1, o0) and np.array_equal(l1, l0)


def test_steady_instance_causal_2k_workload_bit_identical():
    w = inputs.WORKLOADS["bf16_causal_2k"]
    x = workload_inputs("bf16_causal_2k")
    (o1, l1), (o0, l0) = _both(x, causal=w.causal, softmax_scale=w.softmax_scale)
    assert np.array_equal(o1, o0) and np.array_equal(l1, l0)


@pytest.mark.parametrize("causal", [False, True])
def test_steady_instance_varlen(causal):
    # packed sequences: empty query or key ranges, one-block and many-block items
    sq = [5, 0, 130, 1300, 1, 128, 900]
    sk = [7, 3, 0, 1500, 1, 128, 2000]
    x = inputs.make_varlen(sq, sk, heads=3, head_dim=128, seed=29)
    scale = 128 ** -0.5
    (o1, l1), (o0, l0) = _both(x, causal=causal, softmax_scale=scale)
    o_ref, lse_ref = oracle.attention(x["q"], x["k"], x["v"], softmax_scale=scale, causal=causal,
                                      cu_seqlens_q=x["cu_seqlens_q"], cu_seqlens_k=x["cu_seqlens_k"])
    compare(o1, l1, o_ref, lse_ref, what=f"steady instance, varlen causal={causal}")
    assert np.array_equal(o1, o0) and np.array_equal(l1, l0)
