"""The exp2-on-FMA-pipe build option (FA_EXP2_EMU_PAIRS) on the GPU: a library
built with half of every unmasked block's exp2 pairs on the FMA pipe must meet the
same parity bar against the oracle (bf16 and e4m3, causal blocks keep the MUFU)."""
import numpy as np
import pytest

import oracle
import exact_attention_forward_gb300 as fa
from exact_attention_forward_gb300 import _build, inputs
from parity_util import compare, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def emu_library(tmp_path_factory):
    d = tmp_path_factory.mktemp("exp2_fma")
    so = _build.build(force=True, extra_flags=["-DFA_EXP2_EMU_PAIRS=8"],
                      lib_path=str(d / "fa_exp2_fma.so"), build_dir=str(d / "obj"))
    saved_lib, saved_path = fa._lib, fa._LIB_PATH
    fa._lib, fa._LIB_PATH = None, so
    fa.load_library()
    try:
        yield so
    finally:
        fa._lib, fa._LIB_PATH = saved_lib, saved_path


@pytest.mark.parametrize("B,H,Sq,Sk,D,causal", [
    (1, 2, 256, 640, 128, False),
    (2, 2, 384, 384, 128, True),
    (1, 3, 200, 1000, 64, False),
])
def test_bf16_parity_with_fma_exp2(emu_library, B, H, Sq, Sk, D, causal):
    x = inputs.make_random(B, H, Sq, Sk, D, seed=700 + Sq + Sk)
    o, lse = run_gpu(x, causal=causal, softmax_scale=D ** -0.5)
    o_ref, lse_ref = oracle.attention(x["q"], x["k"], x["v"], softmax_scale=D ** -0.5, causal=causal)
    compare(o, lse, o_ref, lse_ref, what=f"fma exp2 {(B, H, Sq, Sk, D, causal)}")


def test_fp8_parity_with_fma_exp2(emu_library):
    w = inputs.Workload("fp8_emu", 1, 2, 256, 512, 128, False, dtype="e4m3", seed=77)
    x = inputs.make_inputs(w)
    o, lse = run_gpu(x, causal=False, softmax_scale=w.softmax_scale)
    o_ref, lse_ref = oracle.attention(x["q"], x["k"], x["v"], softmax_scale=w.softmax_scale,
                                      descale=x["descale"])
    compare(o, lse, o_ref, lse_ref, dtype="e4m3", what="fma exp2 fp8")
