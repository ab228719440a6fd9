"""Parity oracle for the attention forward pass -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The product path (the
``exact_attention_forward_gb300`` package and its CUDA library) never imports,
links or executes anything here, and this package imports nothing from it.

The arithmetic lives in ``attn_oracle.c`` (plain fp64 loops, one query row at
a time, OpenMP over rows).  This module only compiles it with gcc, marshals
arrays and reshapes results.  See the header of ``attn_oracle.c`` for the
definition it follows and the passages it cites.

Every function here is pinned by ``tests/test_oracle_pins.py`` against brute
force, closed forms, invariants and library routines; none is "parity
unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_attn_oracle.so")
# Tests that plant mistakes in the oracle point this at a mutated build (and skip the
# rebuild); nothing else sets it.
_LIB_OVERRIDE = os.environ.get("FA_ORACLE_LIB_OVERRIDE")
_lock = threading.Lock()
_lib = None

DT_F64, DT_BF16, DT_E4M3, DT_E5M2 = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no -ffast-math: fp64 stays IEEE)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(_LIB_OVERRIDE or build())
            lib.orc_attention_rows.restype = ctypes.c_int
            lib.orc_attention_rows.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
            lib.orc_append_kv.restype = ctypes.c_int
            lib.orc_append_kv.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_void_p, ctypes.c_int]
            lib.orc_decode.restype = ctypes.c_int
            lib.orc_decode.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_int64]
            _lib = lib
    return _lib


def _as_storage(x):
    """Return (contiguous numpy array of the raw storage, dtype code)."""
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(x, torch.Tensor):
        x = x.detach().cpu().contiguous()
        if x.dtype == torch.bfloat16:
            return x.view(torch.int16).numpy().view(np.uint16), DT_BF16
        if x.dtype == torch.float8_e4m3fn:
            return x.view(torch.uint8).numpy(), DT_E4M3
        if x.dtype == torch.float8_e5m2:
            return x.view(torch.uint8).numpy(), DT_E5M2
        return x.to(torch.float64).numpy(), DT_F64
    a = np.ascontiguousarray(x)
    if a.dtype == np.float64:
        return a, DT_F64
    return np.ascontiguousarray(a, dtype=np.float64), DT_F64


def decode(x, dtype_code: int) -> np.ndarray:
    """Decode raw bf16 (uint16) or e4m3 / e5m2 (uint8) codes to fp64 with the oracle's decoder."""
    a = np.ascontiguousarray(x)
    out = np.empty(a.shape, dtype=np.float64)
    rc = _load().orc_decode(dtype_code, a.ctypes.data, out.ctypes.data, a.size)
    if rc != 0:
        raise ValueError("bad dtype code")
    return out


def all_rows(batch, heads, seqlen_q=None, seqlens_q=None) -> np.ndarray:
    """(b, h, i) triples for every query row."""
    out = []
    for b in range(batch):
        sq = seqlen_q if seqlens_q is None else int(seqlens_q[b])
        if sq == 0:
            continue
        bb, hh, ii = np.meshgrid([b], np.arange(heads), np.arange(sq), indexing="ij")
        out.append(np.stack([bb.ravel(), hh.ravel(), ii.ravel()], axis=1))
    if not out:
        return np.zeros((0, 3), dtype=np.int64)
    return np.concatenate(out).astype(np.int64)


def _descales(descale, batch, heads_k):
    """Three descales (scalars or arrays broadcastable to [batch, heads_k]) ->
    (three fp64 arrays, stride_b, stride_h) in the oracle's indexing."""
    arrs = [np.asarray(d.cpu().numpy() if hasattr(d, "cpu") else d, dtype=np.float64)
            for d in descale]
    if all(a.size == 1 for a in arrs):
        return [np.ascontiguousarray(a.reshape(1)) for a in arrs], 0, 0
    full = [np.ascontiguousarray(np.broadcast_to(a, (batch, heads_k))) for a in arrs]
    return full, heads_k, 1


def attention_rows(q, k, v, rows, *, softmax_scale, causal=False,
                   cu_seqlens_q=None, cu_seqlens_k=None, seqused_k=None,
                   descale=(1.0, 1.0, 1.0), return_probs=False):
    """Evaluate the given (b, h, i) query rows.

    q, k, v: torch tensors (bf16, float8_e4m3fn, float8_e5m2 or any float ->
    fp64) or numpy arrays, fixed-length [B, S, H, D] or packed [total, H, D]
    with cu_seqlens; K/V may have fewer heads than Q (grouped-query attention)
    and each tensor has its own storage type.  descale: three scalars, or
    arrays broadcastable to [B, Hk] (one value per batch and key/value head).
    seqused_k: optional int [B]; sequence b attends over its first seqused_k[b]
    keys only.
    Returns (O [n, Dv] fp64, LSE [n] fp64[, P [n, max Sk] fp64]).
    """
    qa, dq = _as_storage(q)
    ka, dk = _as_storage(k)
    va, dvt = _as_storage(v)
    varlen = cu_seqlens_q is not None
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    if varlen:
        cq = np.ascontiguousarray(np.asarray(cu_seqlens_q, dtype=np.int32))
        ck = np.ascontiguousarray(np.asarray(cu_seqlens_k, dtype=np.int32))
        batch = cq.size - 1
        heads, d = qa.shape[1], qa.shape[2]
        heads_k = ka.shape[1]
        dv = va.shape[2]
        sq = sk = 0
        max_sk = int(np.max(ck[1:] - ck[:-1])) if batch > 0 else 0
        cq_p, ck_p = cq.ctypes.data, ck.ctypes.data
    else:
        batch, sq, heads, d = qa.shape
        sk = ka.shape[1]
        heads_k = ka.shape[2]
        dv = va.shape[3]
        max_sk = sk
        cq_p = ck_p = None
    n = rows.shape[0]
    o = np.zeros((n, dv), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    p = np.zeros((n, max(max_sk, 1)), dtype=np.float64) if return_probs else None
    ds, ds_b, ds_h = _descales(descale, batch, heads_k)
    used = None
    if seqused_k is not None:
        used = np.ascontiguousarray(np.asarray(
            seqused_k.cpu().numpy() if hasattr(seqused_k, "cpu") else seqused_k, dtype=np.int32))
        if used.shape != (batch,):
            raise ValueError("seqused_k must have one entry per sequence")
    rc = _load().orc_attention_rows(
        qa.ctypes.data, ka.ctypes.data, va.ctypes.data, dq, dk, dvt,
        ds[0].ctypes.data, ds[1].ctypes.data, ds[2].ctypes.data, ds_b, ds_h,
        int(batch), int(heads), int(heads_k), int(sq), int(sk), cq_p, ck_p,
        None if used is None else used.ctypes.data,
        int(d), int(dv), float(softmax_scale), int(bool(causal)),
        rows.ctypes.data, n, o.ctypes.data, lse.ctypes.data,
        None if p is None else p.ctypes.data, 0 if p is None else p.shape[1])
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return (o, lse, p) if return_probs else (o, lse)


def attention(q, k, v, *, softmax_scale, causal=False, cu_seqlens_q=None,
              cu_seqlens_k=None, seqused_k=None, descale=(1.0, 1.0, 1.0)):
    """Every row, returned in the CUDA path's output layouts.

    Fixed length: O [B, Sq, H, Dv], LSE [B, H, Sq].
    Varlen:       O [total_q, H, Dv], LSE [H, total_q].
    """
    varlen = cu_seqlens_q is not None
    if varlen:
        cq = np.asarray(cu_seqlens_q, dtype=np.int64)
        batch = cq.size - 1
        heads = q.shape[1]
        dv = v.shape[2]
        rows = all_rows(batch, heads, seqlens_q=cq[1:] - cq[:-1])
    else:
        batch, sq, heads, _ = q.shape
        dv = v.shape[3]
        rows = all_rows(batch, heads, seqlen_q=sq)
    o_r, lse_r = attention_rows(q, k, v, rows, softmax_scale=softmax_scale, causal=causal,
                                cu_seqlens_q=cu_seqlens_q, cu_seqlens_k=cu_seqlens_k,
                                seqused_k=seqused_k, descale=descale)
    b, h, i = rows[:, 0], rows[:, 1], rows[:, 2]
    if varlen:
        total_q = int(cq[-1])
        o = np.zeros((total_q, heads, dv))
        lse = np.zeros((heads, total_q))
        pos = cq[b] + i
        o[pos, h] = o_r
        lse[h, pos] = lse_r
    else:
        o = np.zeros((batch, sq, heads, dv))
        lse = np.zeros((batch, heads, sq))
        o[b, i, h] = o_r
        lse[b, h, i] = lse_r
    return o, lse


def append_kv(cache, new_rows, seqlens):
    """Return a copy of `cache` [B, capacity, Hk, W] with `new_rows` [B, n_new, Hk, W]
    written at rows seqlens[b] .. seqlens[b] + n_new - 1 of each sequence b
    (bytes copied unchanged; torch bf16 / fp8 tensors come back in their own type,
    other torch floats as fp64)."""
    import torch
    is_t = isinstance(cache, torch.Tensor)
    c = cache.detach().cpu().contiguous().clone() if is_t else np.array(cache, copy=True)
    ca, dt = _as_storage(c)
    na, dn = _as_storage(new_rows)
    if dt != dn:
        raise ValueError("cache and new rows must share one storage type")
    ca = np.ascontiguousarray(ca)
    sl = np.ascontiguousarray(np.asarray(seqlens.cpu().numpy() if hasattr(seqlens, "cpu")
                                         else seqlens, dtype=np.int32))
    batch, cap, hk, w = ca.shape
    n_new = na.shape[1]
    if na.shape != (batch, n_new, hk, w) or sl.shape != (batch,):
        raise ValueError("shape mismatch")
    rc = _load().orc_append_kv(ca.ctypes.data, na.ctypes.data, dt, batch, cap, hk, w,
                               sl.ctypes.data, n_new)
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    if is_t:
        if dt == DT_BF16:
            return torch.from_numpy(ca.view(np.int16)).view(torch.bfloat16)
        if dt == DT_E4M3:
            return torch.from_numpy(ca).view(torch.float8_e4m3fn)
        if dt == DT_E5M2:
            return torch.from_numpy(ca).view(torch.float8_e5m2)
        return torch.from_numpy(ca)  # any other float type comes back as fp64
    return ca


def merge_partials(o_parts, lse_parts):
    """Merge attention results over disjoint key chunks by the log-sum-exp identity.

    LSE = ln sum_c exp(LSE_c);  O = sum_c exp(LSE_c - LSE) O_c.
    Chunks with LSE_c = -inf contribute nothing; all -inf -> O = 0, LSE = -inf.
    """
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    o_parts = np.asarray(o_parts, dtype=np.float64)
    m = np.max(lse_parts, axis=0)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    w = np.exp(lse_parts - m_safe)
    tot = np.sum(w, axis=0)
    with np.errstate(divide="ignore"):
        lse = np.where(tot > 0, m_safe + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
    wn = np.where(tot > 0, w / np.where(tot > 0, tot, 1.0), 0.0)
    o = np.sum(wn[..., None] * o_parts, axis=0)
    return o, lse
