"""The entry point that allocates nothing: fa_fwd_static_workspace (GPU).

It serves callers that cannot call cudaMalloc: code running inside a host
program that owns all device memory and hands out no scratch, and
latency-critical loops where cudaMalloc / cudaFree would synchronise the
device.  When the shape splits its key range, the partial results go to a
fixed 16 MiB array inside the library instead of a caller workspace.

Here it is called through the C ABI and checked against fa_fwd with a caller
workspace, on two calls in a row with different inputs (the second call finds
the first call's partials still in the shared array), plus the rejection of a
shape whose split scratch would not fit.  This file sorts last so that a run
that stops at the first failure has run every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

import exact_attention_forward_gb300 as fa
from exact_attention_forward_gb300 import inputs
from parity_util import compare

pytestmark = pytest.mark.gpu

STATIC_BYTES = 16 << 20


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return fa.load_library()


def _call_static(lib, q, k, v, o, lse, causal):
    b, sq, h, d = q.shape
    sk = k.shape[1]
    stream = torch.cuda.current_stream()
    return lib.fa_fwd_static_workspace(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                       lse.data_ptr(), b, h, sq, sk, d, d, float(d ** -0.5),
                                       int(causal), fa.FA_DTYPE_BF16, None, None, None,
                                       ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("causal", [False, True])
def test_static_workspace_matches_fa_fwd_on_two_calls(lib, causal):
    w = inputs.WORKLOADS["bf16_shortq_longkv"]  # B=1 H=8 Sq=128 Sk=65536: splits the keys
    need = fa.workspace_size(w.batch, w.heads, w.seqlen_q, w.seqlen_k, w.head_dim, causal)
    assert 0 < need <= STATIC_BYTES
    for call, seed in enumerate((w.seed, w.seed + 17)):
        x = inputs.make_inputs(w, seed=seed)
        q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
        o_ref, lse_ref = fa.fwd(q, k, v, causal=causal, softmax_scale=w.softmax_scale,
                                workspace="auto")
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        st = _call_static(lib, q, k, v, o, lse, causal)
        assert st == fa.FA_OK, lib.fa_last_error_detail()
        torch.cuda.synchronize()
        assert fa.device_error(clear=True)[0] == fa.FA_OK
        compare(o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
                o_ref.float().cpu().numpy().astype(np.float64),
                lse_ref.cpu().numpy().astype(np.float64), what=f"static workspace call {call}")


def test_static_workspace_rejects_shapes_that_do_not_fit(lib):
    b, h, sq, sk, d = 1, 4, 2048, 65536, 128
    assert fa.workspace_size(b, h, sq, sk, d) > STATIC_BYTES
    x = inputs.make_random(b, h, sq, sk, d, seed=5)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o = torch.full((b, sq, h, d), 3.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((b, h, sq), 5.0, dtype=torch.float32, device="cuda")
    st = _call_static(lib, q, k, v, o, lse, False)
    assert st == fa.FA_ERR_WORKSPACE
    assert b"needed" in lib.fa_last_error_detail()
    torch.cuda.synchronize()
    assert torch.all(o == 3.0) and torch.all(lse == 5.0)
