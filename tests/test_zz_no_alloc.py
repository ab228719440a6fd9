"""The entry point that allocates nothing: fa_fwd_static_workspace (GPU).

It serves callers that cannot call cudaMalloc: code running inside a host
program that owns all device memory and hands out no scratch, and
latency-critical loops where cudaMalloc / cudaFree would synchronise the
device.  When the shape splits its key range, the partial results go to a
fixed 16 MiB array inside the library instead of a caller workspace.

Here it is called through the C ABI, twice in a row on different inputs, the
second call splitting the key range fewer ways than the first (so partial rows
the first call left in the shared array would show if they were merged).  Each
call must be bit-identical to fa_fwd with a caller workspace -- the same
kernels and the same split count -- and within the parity bounds of the fp64
oracle.  The rejection of a shape whose split scratch would not fit is checked
too.  This file sorts last so that a run that stops at the first failure has
run every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import exact_attention_forward_gb300 as fa
from exact_attention_forward_gb300 import inputs
from parity_util import compare, nan_outputs

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
    # B=1 H=8 Sq=128: 65536 keys split 19 ways, then 4096 keys split 8 ways
    B, H, Sq, D = 1, 8, 128, 128
    splits_seen = []
    for call, (sk, seed) in enumerate(((65536, 1006), (4096, 1023))):
        splits = fa.num_splits(B, H, Sq, sk, causal)
        need = fa.workspace_size(B, H, Sq, sk, D, causal)
        assert splits > 1 and 0 < need <= STATIC_BYTES
        splits_seen.append(splits)
        x = inputs.make_random(B, H, Sq, sk, D, seed=seed)
        q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
        # fa_fwd with a caller-owned workspace of the size it asks for
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        o_ws, lse_ws = nan_outputs(q, v, (B, H, Sq))
        fa.fwd(q, k, v, causal=causal, softmax_scale=D ** -0.5, workspace=ws, out=o_ws,
               lse=lse_ws)
        o, lse = nan_outputs(q, v, (B, H, Sq))
        st = _call_static(lib, q, k, v, o, lse, causal)
        assert st == fa.FA_OK, lib.fa_last_error_detail()
        torch.cuda.synchronize()
        assert fa.device_error(clear=True)[0] == fa.FA_OK
        # same kernels, same splits: the same bits
        assert torch.equal(o.view(torch.int16), o_ws.view(torch.int16)), f"call {call}: O differs"
        assert torch.equal(lse.view(torch.int32), lse_ws.view(torch.int32)), f"call {call}: LSE differs"
        o_ref, lse_ref = oracle.attention(x["q"], x["k"], x["v"], softmax_scale=D ** -0.5,
                                          causal=causal)
        compare(o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
                o_ref, lse_ref, what=f"static workspace call {call} (causal={causal})")
    assert splits_seen[1] < splits_seen[0]


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
