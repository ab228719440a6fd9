"""CPU-only checks of the CUDA library: it builds, loads without a GPU and
exports every function include/fa.h declares; argument validation that runs
before any device work returns the documented codes."""
import ctypes
import os
import re

import pytest

import exact_attention_forward_gb300 as fa
from exact_attention_forward_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return fa.load_library()


def header_functions():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert header_functions() == sorted(fa.EXPORTED_SYMBOLS)


def test_every_declared_symbol_is_exported(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_status_strings(lib):
    for code in range(7):
        assert lib.fa_status_string(code)
    assert b"unknown" in lib.fa_status_string(99)


# a fake, 16-byte aligned address: validation never dereferences pointers
P = ctypes.c_void_p(0x10000)


def call(lib, **kw):
    a = dict(q=P, k=P, v=P, o=P, lse=P, batch=1, heads=1, sq=128, sk=128, cuq=None, cuk=None,
             mq=0, mk=0, d=128, dv=128, scale=0.1, causal=0, dtype=0, qd=None, kd=None, vd=None,
             ws=None, wsb=0, stream=None)
    a.update(kw)
    return lib.fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["batch"], a["heads"], a["sq"],
                      a["sk"], a["cuq"], a["cuk"], a["mq"], a["mk"], a["d"], a["dv"], a["scale"],
                      a["causal"], a["dtype"], a["qd"], a["kd"], a["vd"], a["ws"], a["wsb"],
                      a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(o=ctypes.c_void_p(0x10008)), fa.FA_ERR_INVALID_ARG),
    (dict(heads=0), fa.FA_ERR_INVALID_ARG),
    (dict(batch=-1), fa.FA_ERR_INVALID_ARG),
    (dict(sq=-5), fa.FA_ERR_INVALID_ARG),
    (dict(causal=2), fa.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(dtype=7), fa.FA_ERR_INVALID_ARG),
    (dict(qd=P), fa.FA_ERR_INVALID_ARG),             # descale with bf16
    (dict(cuq=P), fa.FA_ERR_INVALID_ARG),            # only one cu_seqlens
    (dict(d=96, dv=96), fa.FA_ERR_UNSUPPORTED),
    (dict(d=128, dv=64), fa.FA_ERR_UNSUPPORTED),
    (dict(d=64, dv=64, dtype=1), fa.FA_ERR_UNSUPPORTED),
])
def test_validation_codes(lib, kw, code):
    assert call(lib, **kw) == code
    assert lib.fa_last_error_detail()


def test_empty_problems_are_ok_without_a_device(lib):
    assert call(lib, batch=0) == fa.FA_OK
    assert call(lib, sq=0) == fa.FA_OK


def test_gqa_validation(lib):
    def gqa(heads, heads_k):
        return lib.fa_fwd_gqa(P, P, P, P, P, 1, heads, heads_k, 128, 128, None, None, 0, 0, 128,
                              128, 0.1, 0, 0, None, None, None, None, 0, None)
    assert gqa(8, 3) == fa.FA_ERR_INVALID_ARG   # 3 does not divide 8
    assert gqa(8, 0) == fa.FA_ERR_INVALID_ARG
    assert gqa(8, 16) == fa.FA_ERR_INVALID_ARG
    assert b"heads_k" in lib.fa_last_error_detail()


def fp8(lib, **kw):
    a = dict(batch=1, heads=4, heads_k=2, sq=128, sk=128, d=128, vdt=fa.FA_DTYPE_E5M2, qd=P, kd=P,
             vd=P, sb=2, sh=1)
    a.update(kw)
    return lib.fa_fwd_fp8(P, P, P, P, P, a["batch"], a["heads"], a["heads_k"], a["sq"], a["sk"],
                          None, None, 0, 0, a["d"], 0.1, 0, a["vdt"], a["qd"], a["kd"], a["vd"],
                          a["sb"], a["sh"], None, 0, None)


@pytest.mark.parametrize("kw,code", [
    (dict(vdt=fa.FA_DTYPE_BF16), fa.FA_ERR_INVALID_ARG),    # V type must be an FP8 type
    (dict(vdt=9), fa.FA_ERR_INVALID_ARG),
    (dict(sb=-1), fa.FA_ERR_INVALID_ARG),                   # negative descale stride
    (dict(qd=ctypes.c_void_p(0x10002)), fa.FA_ERR_INVALID_ARG),  # misaligned descale
    (dict(heads_k=3), fa.FA_ERR_INVALID_ARG),
    (dict(d=64), fa.FA_ERR_UNSUPPORTED),
])
def test_fp8_validation(lib, kw, code):
    assert fp8(lib, **kw) == code
    assert lib.fa_last_error_detail()


def test_fp8_empty_problem_is_ok_without_a_device(lib):
    assert fp8(lib, batch=0) == fa.FA_OK


def test_e5m2_only_accepted_for_v(lib):
    # fa_fwd_gqa takes one type for q, k and v: E5M2 is not one of them
    assert lib.fa_fwd_gqa(P, P, P, P, P, 1, 2, 2, 128, 128, None, None, 0, 0, 128, 128, 0.1, 0,
                          fa.FA_DTYPE_E5M2, None, None, None, None, 0, None) == fa.FA_ERR_INVALID_ARG


def kvc(lib, **kw):
    a = dict(kc=P, vc=P, kn=P, vn=P, batch=2, heads=4, heads_k=2, sq=1, cap=4096, lens=P, n_new=1,
             d=128, dt=fa.FA_DTYPE_BF16, vdt=fa.FA_DTYPE_BF16, qd=None)
    a.update(kw)
    return lib.fa_fwd_kvcache(P, a["kc"], a["vc"], a["kn"], a["vn"], P, P, a["batch"], a["heads"],
                              a["heads_k"], a["sq"], a["cap"], a["lens"], a["n_new"], a["d"], 0.1,
                              1, a["dt"], a["vdt"], a["qd"], None, None, 0, 0, None, 0, None)


@pytest.mark.parametrize("kw,code", [
    (dict(kc=None), fa.FA_ERR_INVALID_ARG),
    (dict(lens=None), fa.FA_ERR_INVALID_ARG),
    (dict(lens=ctypes.c_void_p(0x10002)), fa.FA_ERR_INVALID_ARG),
    (dict(kn=None), fa.FA_ERR_INVALID_ARG),            # new rows announced but not given
    (dict(vn=ctypes.c_void_p(0x10008)), fa.FA_ERR_INVALID_ARG),
    (dict(n_new=-1), fa.FA_ERR_INVALID_ARG),
    (dict(n_new=5000), fa.FA_ERR_INVALID_ARG),         # more new rows than the capacity
    (dict(cap=0), fa.FA_ERR_INVALID_ARG),
    (dict(vdt=fa.FA_DTYPE_E5M2), fa.FA_ERR_INVALID_ARG),  # bf16 q/k with an FP8 V
    (dict(qd=P), fa.FA_ERR_INVALID_ARG),               # descale with bf16
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
])
def test_kvcache_validation(lib, kw, code):
    assert kvc(lib, **kw) == code
    assert lib.fa_last_error_detail()


def test_kvcache_empty_batch_is_ok_without_a_device(lib):
    assert kvc(lib, batch=0) == fa.FA_OK


def pair(lib, **kw):
    a = dict(batch=1, heads=4, heads_k=2, sq=128, sk=128, d=128, scale=0.1, causal=1, q=P)
    a.update(kw)
    return lib.fa_fwd_2cta(a["q"], P, P, P, P, a["batch"], a["heads"], a["heads_k"], a["sq"],
                           a["sk"], None, None, 0, 0, a["d"], a["scale"], a["causal"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(heads_k=3), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-1.0), fa.FA_ERR_INVALID_ARG),
    (dict(causal=3), fa.FA_ERR_INVALID_ARG),
    (dict(d=64), fa.FA_ERR_UNSUPPORTED),               # the CTA-pair kernel is built for D = 128
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
])
def test_cta_pair_validation(lib, kw, code):
    assert pair(lib, **kw) == code
    assert lib.fa_last_error_detail()


def test_cta_pair_empty_problem_is_ok_without_a_device(lib):
    assert pair(lib, batch=0) == fa.FA_OK


def test_static_workspace_without_a_device_says_why(lib):
    # with no usable device the entry point that allocates nothing fails before any device
    # work, with FA_ERR_CUDA and a detail message (never a stale or empty one)
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present: this checks the no-device path")
    lib.fa_fwd(None, P, P, P, P, 1, 1, 128, 128, None, None, 0, 0, 128, 128, 0.1, 0, 0,
               None, None, None, None, 0, None)  # leaves an unrelated detail behind
    st = lib.fa_fwd_static_workspace(P, P, P, P, P, 1, 1, 128, 128, 128, 128, 0.1, 0, 0,
                                     None, None, None, None)
    assert st == fa.FA_ERR_CUDA
    detail = lib.fa_last_error_detail()
    assert b"no usable current CUDA device" in detail or b"static scratch" in detail, detail


def test_microbench_library_exports_its_header():
    text = open(os.path.join(ROOT, "include", "fa_microbench.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = sorted(set(re.findall(r"\b(fa_mb_[a-z0-9_]+)\s*\(", text)))
    assert names == ["fa_mb_ex2", "fa_mb_ex2_f16x2", "fa_mb_ex2_per_cta", "fa_mb_load", "fa_mb_load_bytes_per_cta",
                     "fa_mb_mma", "fa_mb_mma_flops_per_cta", "fa_mb_mma_with_load"]
    mb = ctypes.CDLL(_build.build_microbench())
    for name in names:
        assert isinstance(getattr(mb, name), ctypes._CFuncPtr)
    mb.fa_mb_mma_flops_per_cta.restype = ctypes.c_longlong
    mb.fa_mb_ex2_per_cta.restype = ctypes.c_longlong
    # 4 MMAs of 2 * 128 * N * K per iteration; 1024 threads x 8 chains x 4 per iteration
    assert mb.fa_mb_mma_flops_per_cta(256, 0, 10) == 4 * 10 * 2 * 128 * 256 * 16
    assert mb.fa_mb_mma_flops_per_cta(128, 1, 10) == 4 * 10 * 2 * 128 * 128 * 32
    assert mb.fa_mb_ex2_per_cta(10) == 1024 * 8 * 4 * 10
    mb.fa_mb_load_bytes_per_cta.restype = ctypes.c_longlong
    assert mb.fa_mb_load_bytes_per_cta(10) == 10 * 32 * 1024


def test_trace_is_unsupported_in_the_default_build(lib):
    # the default library holds no trace code: asking for a trace says so
    assert lib.fa_debug_trace(None, 0) == fa.FA_ERR_UNSUPPORTED
    assert b"FA_TRACE" in lib.fa_last_error_detail()
    assert lib.fa_debug_trace_bytes() == 8 * 4 * 8192 * 8
