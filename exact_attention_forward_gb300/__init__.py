"""Attention forward pass for one GB300 (sm_103a) -- Python binding.

Every step of the computation runs in the CUDA library ``_fa_gb300.so``
(built from ``csrc/`` by ``_build.py``) behind the C ABI of ``include/fa.h``.
This module only marshals arguments: it takes torch tensors for device memory
and streams, allocates outputs with torch, and calls ``fa_fwd`` through
ctypes.  There is no fallback: if the library is missing or the call fails,
it raises.

    o, lse = fwd(q, k, v, causal=True)

q, k, v: CUDA tensors, bf16 or float8_e4m3fn (v may be float8_e5m2 with
e4m3 q/k), [B, S, H, D] (or packed [total, H, D] with cu_seqlens_q /
cu_seqlens_k int32 [B + 1] on the device); k and v may have fewer heads than
q (grouped-query attention).  FP8 descales are scalars or one value per
(batch, K/V head).  Returns o (bf16, q's layout) and lse (fp32, [B, H, Sq] or
[H, total_q]).

    o, lse = fwd_kvcache(q, k_cache, v_cache, cache_seqlens, k_new, v_new, causal=True)

appends k_new / v_new to the caches at cache_seqlens and attends over the
first cache_seqlens + seqlen_new rows of each sequence.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

__all__ = ["fwd", "fwd_kvcache", "fa_fwd", "FaError", "workspace_size", "num_splits",
           "kvcache_workspace_size", "kvcache_num_splits",
           "device_error", "debug_set", "debug_select_steady", "library_path", "EXPORTED_SYMBOLS", "load_library"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_fa_gb300.so")

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_WORKSPACE, \
    FA_ERR_DEVICE_TIMEOUT, FA_ERR_DEVICE_ARG = range(7)
FA_DTYPE_BF16, FA_DTYPE_E4M3, FA_DTYPE_E5M2 = 0, 1, 2

# Every function declared in include/fa.h.
EXPORTED_SYMBOLS = ("fa_fwd", "fa_fwd_workspace_size", "fa_fwd_num_splits", "fa_status_string",
                    "fa_last_error_detail", "fa_device_error", "fa_debug_set",
                    "fa_fwd_static_workspace", "fa_fwd_gqa", "fa_fwd_fp8", "fa_fwd_kvcache",
                    "fa_fwd_workspace_size_gqa", "fa_fwd_num_splits_gqa", "fa_fwd_2cta",
                    "fa_fwd_kvcache_workspace_size", "fa_fwd_kvcache_num_splits",
                    "fa_debug_trace", "fa_debug_trace_bytes", "fa_debug_select_steady")

_lock = threading.Lock()
_lib = None


class FaError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"fa_fwd failed: status {status} ({detail})")
        self.status = status
        self.detail = detail


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"CUDA extension {_LIB_PATH} is missing; build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.fa_fwd.restype = i32
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, i32, i32, i32, i32,
                               f32, i32, i32, vp, vp, vp, vp, sz, vp]
        lib.fa_fwd_workspace_size.restype = sz
        lib.fa_fwd_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
        lib.fa_fwd_num_splits.restype = i32
        lib.fa_fwd_num_splits.argtypes = [i32, i32, i32, i32, i32]
        lib.fa_fwd_workspace_size_gqa.restype = sz
        lib.fa_fwd_workspace_size_gqa.argtypes = [i32, i32, i32, i32, i32, i32, i32]
        lib.fa_fwd_num_splits_gqa.restype = i32
        lib.fa_fwd_num_splits_gqa.argtypes = [i32, i32, i32, i32, i32, i32]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_status_string.argtypes = [i32]
        lib.fa_last_error_detail.restype = ctypes.c_char_p
        lib.fa_last_error_detail.argtypes = []
        lib.fa_device_error.restype = i32
        lib.fa_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
        lib.fa_debug_set.restype = None
        lib.fa_debug_set.argtypes = [ctypes.c_uint64, ctypes.c_uint32]
        lib.fa_debug_select_steady.restype = None
        lib.fa_debug_select_steady.argtypes = [i32]
        lib.fa_debug_trace.restype = i32
        lib.fa_debug_trace.argtypes = [vp, sz]
        lib.fa_debug_trace_bytes.restype = sz
        lib.fa_debug_trace_bytes.argtypes = []
        lib.fa_fwd_gqa.restype = i32
        lib.fa_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, i32, i32,
                                   i32, i32, f32, i32, i32, vp, vp, vp, vp, sz, vp]
        i64 = ctypes.c_int64
        lib.fa_fwd_fp8.restype = i32
        lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, i32, i32,
                                   i32, f32, i32, i32, vp, vp, vp, i64, i64, vp, sz, vp]
        lib.fa_fwd_kvcache.restype = i32
        lib.fa_fwd_kvcache.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp,
                                       i32, i32, f32, i32, i32, i32, vp, vp, vp, i64, i64, vp, sz,
                                       vp]
        lib.fa_fwd_kvcache_workspace_size.restype = sz
        lib.fa_fwd_kvcache_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
        lib.fa_fwd_kvcache_num_splits.restype = i32
        lib.fa_fwd_kvcache_num_splits.argtypes = [i32, i32, i32, i32, i32, i32]
        lib.fa_fwd_2cta.restype = i32
        lib.fa_fwd_2cta.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, i32, i32,
                                    i32, f32, i32, vp]
        lib.fa_fwd_static_workspace.restype = i32
        lib.fa_fwd_static_workspace.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32,
                                                f32, i32, i32, vp, vp, vp, vp]
        _lib = lib
        return lib


def _detail(lib) -> str:
    d = lib.fa_last_error_detail()
    return d.decode() if d else ""


def fa_fwd(*args) -> int:
    """Raw call of the C entry point (arguments exactly as in include/fa.h)."""
    return load_library().fa_fwd(*args)


def workspace_size(batch, heads, seqlen_q, seqlen_k, head_dim_v, causal=False, heads_k=None) -> int:
    return int(load_library().fa_fwd_workspace_size_gqa(
        batch, heads, heads if heads_k is None else heads_k, seqlen_q, seqlen_k, head_dim_v,
        int(bool(causal))))


def kvcache_workspace_size(batch, heads, heads_k, seqlen_q, cache_capacity, head_dim,
                           causal=False) -> int:
    return int(load_library().fa_fwd_kvcache_workspace_size(
        batch, heads, heads_k, seqlen_q, cache_capacity, head_dim, int(bool(causal))))


def kvcache_num_splits(batch, heads, heads_k, seqlen_q, cache_capacity, causal=False) -> int:
    return int(load_library().fa_fwd_kvcache_num_splits(
        batch, heads, heads_k, seqlen_q, cache_capacity, int(bool(causal))))


def num_splits(batch, heads, seqlen_q, seqlen_k, causal=False, heads_k=None) -> int:
    return int(load_library().fa_fwd_num_splits_gqa(
        batch, heads, heads if heads_k is None else heads_k, seqlen_q, seqlen_k,
        int(bool(causal))))


def device_error(clear: bool = True):
    """(status, flags) of the device-side failure word; see fa_device_error."""
    lib = load_library()
    flags = ctypes.c_uint32(0)
    st = lib.fa_device_error(ctypes.byref(flags), int(bool(clear)))
    return st, flags.value


def debug_set(wait_limit_ns: int = 0, inject: int = 0) -> None:
    load_library().fa_debug_set(int(wait_limit_ns), int(inject))


def debug_select_steady(mode: int = 0) -> None:
    """Kernel instance of bf16 head_dim-128 launches without a cache: 0 by size (default),
    1 always the steady-block instance, -1 never (fa_debug_select_steady)."""
    load_library().fa_debug_select_steady(int(mode))


def _ptr(t):
    return None if t is None else t.data_ptr()


def _fp8_descales(descale, batch, heads_k, dev, temps):
    """(q, k, v) descales -> three fp32 CUDA tensors (or None) and the (batch, head)
    strides of the C ABI: all scalars -> 0-d tensors, strides (0, 0); otherwise every
    descale becomes a contiguous [batch, heads_k] tensor, strides (heads_k, 1)."""
    import torch

    if descale is None:
        return [None, None, None], 0, 0
    per_head = any(isinstance(x, torch.Tensor) and x.numel() > 1 for x in descale)
    out = []
    for x in descale:
        if x is None and not per_head:
            out.append(None)
            continue
        if x is None:
            x = 1.0
        if not isinstance(x, torch.Tensor):
            x = torch.tensor(float(x), dtype=torch.float32, device=dev)
            temps.append(x)
        if per_head:
            y = x.to(device=dev, dtype=torch.float32).expand(batch, heads_k).contiguous()
            if y is not x:
                temps.append(y)
            x = y
        elif x.dtype != torch.float32 or x.device != dev:  # one value: move it over
            x = x.to(device=dev, dtype=torch.float32).reshape(())
            temps.append(x)
        out.append(x)
    return out, (heads_k if per_head else 0), (1 if per_head else 0)


def fwd(q, k, v, *, causal=False, softmax_scale=None, cu_seqlens_q=None, cu_seqlens_k=None,
        max_seqlen_q=None, max_seqlen_k=None, descale=None, workspace="auto", out=None,
        lse=None, stream=None, cta_pair=False):
    """Attention forward on the current CUDA device.  Returns (o, lse).

    descale: for FP8 inputs, (q, k, v) descales as python floats, 0-d fp32 CUDA
    tensors, or fp32 CUDA tensors of shape [B, Hk] (one value per batch and K/V
    head) (None = 1.0).  v may be float8_e5m2 when q and k are float8_e4m3fn.
    workspace: "auto" (allocated with torch when the shape benefits from
    splitting the key range), None (never split) or a caller-owned uint8 CUDA
    tensor.
    cta_pair: run the CTA-pair kernel (fa_fwd_2cta: bf16, head dim 128, no key
    splits; the workspace argument is then unused).
    """
    import torch

    lib = load_library()
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if q.dtype == torch.bfloat16:
        dt = FA_DTYPE_BF16
    elif q.dtype == torch.float8_e4m3fn:
        dt = FA_DTYPE_E4M3
    else:
        raise ValueError(f"unsupported dtype {q.dtype}")
    v_e5m2 = dt == FA_DTYPE_E4M3 and v.dtype == torch.float8_e5m2
    if k.dtype != q.dtype or (v.dtype != q.dtype and not v_e5m2):
        raise ValueError("q, k, v must share one dtype (or be e4m3, e4m3, e5m2)")
    varlen = cu_seqlens_q is not None
    heads_k = k.shape[-2]
    if varlen:
        total_q, heads, d = q.shape
        total_k = k.shape[0]
        dv = v.shape[2]
        batch = cu_seqlens_q.numel() - 1
        if max_seqlen_q is None or max_seqlen_k is None:
            raise ValueError("varlen needs max_seqlen_q and max_seqlen_k")
        sq_arg, sk_arg = total_q, total_k
        o_shape = (total_q, heads, dv)
        lse_shape = (heads, total_q)
        mq, mk = int(max_seqlen_q), int(max_seqlen_k)
    else:
        batch, sq, heads, d = q.shape
        sk = k.shape[1]
        dv = v.shape[3]
        sq_arg, sk_arg = sq, sk
        o_shape = (batch, sq, heads, dv)
        lse_shape = (batch, heads, sq)
        mq, mk = sq, sk
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    dev = q.device
    if out is None:
        out = torch.empty(o_shape, dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty(lse_shape, dtype=torch.float32, device=dev)
    ds = [None, None, None]
    ds_b = ds_h = 0
    temps = []  # tensors made here that must outlive the kernel on `stream`
    if dt == FA_DTYPE_E4M3:
        ds, ds_b, ds_h = _fp8_descales(descale, batch, heads_k, dev, temps)
    ws = None
    ws_bytes = 0
    if cta_pair:
        workspace = None
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError('workspace must be "auto", None or a uint8 CUDA tensor')
        # (varlen: sized by the longest sequences)
        need = workspace_size(batch, heads, mq, mk, dv, causal, heads_k=heads_k) if mq > 0 else 0
        if need > 0:  # allocated from torch's caching allocator (no cudaMalloc per call)
            ws = torch.empty(need, dtype=torch.uint8, device=dev)
            ws_bytes = need
            temps.append(ws)
    elif workspace is not None:
        ws = workspace
        ws_bytes = workspace.numel() * workspace.element_size()
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    if cta_pair:
        if dt != FA_DTYPE_BF16 or d != dv:
            raise ValueError("cta_pair needs bf16 inputs with head_dim == head_dim_v")
        st = lib.fa_fwd_2cta(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), int(batch),
                             int(heads), int(heads_k), int(sq_arg), int(sk_arg),
                             _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), mq, mk, int(d),
                             float(softmax_scale), int(bool(causal)),
                             ctypes.c_void_p(stream.cuda_stream))
    elif dt == FA_DTYPE_E4M3 and (v_e5m2 or ds_b or ds_h):
        if d != dv:
            raise ValueError("FP8 needs head_dim == head_dim_v")
        st = lib.fa_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), int(batch),
                            int(heads), int(heads_k), int(sq_arg), int(sk_arg),
                            _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), mq, mk, int(d),
                            float(softmax_scale), int(bool(causal)),
                            FA_DTYPE_E5M2 if v_e5m2 else FA_DTYPE_E4M3,
                            _ptr(ds[0]), _ptr(ds[1]), _ptr(ds[2]), ds_b, ds_h, _ptr(ws), ws_bytes,
                            ctypes.c_void_p(stream.cuda_stream))
    else:
        st = lib.fa_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), int(batch),
                            int(heads), int(heads_k), int(sq_arg), int(sk_arg), _ptr(cu_seqlens_q),
                            _ptr(cu_seqlens_k), mq, mk, int(d), int(dv), float(softmax_scale),
                            int(bool(causal)), dt, _ptr(ds[0]), _ptr(ds[1]), _ptr(ds[2]), _ptr(ws),
                            ws_bytes, ctypes.c_void_p(stream.cuda_stream))
    if st != FA_OK:
        raise FaError(st, _detail(lib))
    for t in temps:
        t.record_stream(stream)
    return out, lse


def fwd_kvcache(q, k_cache, v_cache, cache_seqlens, k_new=None, v_new=None, *, causal=False,
                softmax_scale=None, descale=None, workspace="auto", out=None, lse=None,
                stream=None):
    """Append k_new / v_new ([B, S_new, Hk, D]) to the caches ([B, capacity, Hk, D],
    written in place) at rows cache_seqlens[b] (int32 CUDA [B], not modified), then
    attend q ([B, Sq, H, D]) over the first cache_seqlens[b] + S_new rows of each
    sequence (causal: bottom-right aligned).  Returns (o [B, Sq, H, D] bf16,
    lse [B, H, Sq] fp32).  Types and descales as fwd()."""
    import torch

    lib = load_library()
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache),
                    ("cache_seqlens", cache_seqlens), ("k_new", k_new), ("v_new", v_new)):
        if t is None:
            continue
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if cache_seqlens.dtype != torch.int32:
        raise ValueError("cache_seqlens must be int32")
    if (k_new is None) != (v_new is None):
        raise ValueError("give both k_new and v_new, or neither")
    if q.dtype == torch.bfloat16:
        dt = vdt = FA_DTYPE_BF16
    elif q.dtype == torch.float8_e4m3fn:
        dt = FA_DTYPE_E4M3
        vdt = FA_DTYPE_E5M2 if v_cache.dtype == torch.float8_e5m2 else FA_DTYPE_E4M3
    else:
        raise ValueError(f"unsupported dtype {q.dtype}")
    batch, sq, heads, d = q.shape
    _, cap, heads_k, _ = k_cache.shape
    n_new = 0 if k_new is None else k_new.shape[1]
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    dev = q.device
    if out is None:
        out = torch.empty((batch, sq, heads, d), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((batch, heads, sq), dtype=torch.float32, device=dev)
    temps = []
    ds, ds_b, ds_h = ([None, None, None], 0, 0)
    if dt == FA_DTYPE_E4M3:
        ds, ds_b, ds_h = _fp8_descales(descale, batch, heads_k, dev, temps)
    ws, ws_bytes = None, 0
    if isinstance(workspace, str):
        need = kvcache_workspace_size(batch, heads, heads_k, sq, cap, d, causal) if sq > 0 else 0
        if need > 0:
            ws = torch.empty(need, dtype=torch.uint8, device=dev)
            ws_bytes = need
            temps.append(ws)
    elif workspace is not None:
        ws = workspace
        ws_bytes = workspace.numel() * workspace.element_size()
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    st = lib.fa_fwd_kvcache(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new),
                            _ptr(out), _ptr(lse), int(batch), int(heads), int(heads_k), int(sq),
                            int(cap), _ptr(cache_seqlens), int(n_new), int(d),
                            float(softmax_scale), int(bool(causal)), dt, vdt, _ptr(ds[0]),
                            _ptr(ds[1]), _ptr(ds[2]), ds_b, ds_h, _ptr(ws), ws_bytes,
                            ctypes.c_void_p(stream.cuda_stream))
    if st != FA_OK:
        raise FaError(st, _detail(lib))
    for t in temps:
        t.record_stream(stream)
    return out, lse
