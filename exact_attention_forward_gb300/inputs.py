"""Seeded synthetic inputs for the attention forward pass.

This module holds input generation only -- random draws, casts to the
storage dtype, per-tensor FP8 quantisation and varlen length draws -- and no
attention arithmetic.  Tests feed the same bytes to the CUDA path and to the
oracle; the benchmark uses the same recipes.

Workloads (shapes and value distributions of the attention configurations):
  bf16_small          B=1  H=2  S=256          D=64   N(0,1)     non-causal  seed 1001
  bf16_causal_2k      B=4  H=16 S=2048         D=128  N(0,1)     causal      seed 1002
  bf16_causal_8k      B=2  H=32 S=8192         D=128  2*N(0,1)   causal      seed 1003
  bf16_noncausal_8k   B=2  H=32 S=8192         D=128  2*N(0,1)   non-causal  seed 1003
  bf16_varlen_causal  16 seqs, S~U{1..4096}, +2 with Sk=0; H=16 D=128 causal seed 1004
  fp8_noncausal_4k    B=4  H=16 S=4096 D=128 e4m3 per-tensor amax/448  non-causal seed 1005
  bf16_shortq_longkv  B=1  H=8  Sq=128 Sk=65536 D=128 N(0,1) non-causal  seed 1006
  bf16_gqa_causal_8k  B=2  H=32 (8 K/V heads) S=8192 D=128 2*N(0,1) causal seed 1007
  fp8_headscale_4k    B=4  H=16 S=4096 D=128 Q/K e4m3, V e5m2, one descale per
                      (batch, head) = amax/max-finite       non-causal  seed 1008
  bf16_kvcache_decode B=16 H=32 (8 K/V heads) D=128, a K/V cache of capacity 8192
                      filled to U{4096..8191} rows per sequence; one new token
                      (q, k_new, v_new of 1 row) appended, then attended   seed 1009
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

E4M3_MAX = 448.0
E5M2_MAX = 57344.0
_FP8 = {"e4m3": (torch.float8_e4m3fn, E4M3_MAX), "e5m2": (torch.float8_e5m2, E5M2_MAX)}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    heads: int
    seqlen_q: int
    seqlen_k: int
    head_dim: int
    causal: bool
    dtype: str = "bf16"          # "bf16" or "e4m3" (the type of Q and K, and of V by default)
    v_dtype: str = ""            # "e5m2" to store V as E5M2 (FP8 only); "" = dtype
    descale: str = "tensor"      # FP8: "tensor" (one descale per tensor) or "head" (per batch, K/V head)
    amp: float = 1.0             # values are amp * N(0,1)
    seed: int = 0
    varlen: bool = False         # lengths drawn per sequence (seqlen_q/k = max 4096)
    n_seqs: int = 0
    empty_k_at: tuple = ()       # packed positions of sequences with seqlen_k = 0
    heads_k: int = 0             # K/V heads (grouped-query attention); 0 = heads
    cache_new: int = 0           # > 0: K/V cache workload; seqlen_k is the cache capacity,
                                 #   seqlen_q = cache_new new rows are appended, then attended

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def kv_heads(self) -> int:
        return self.heads_k or self.heads


WORKLOADS = {
    "bf16_small": Workload("bf16_small", 1, 2, 256, 256, 64, False, seed=1001),
    "bf16_causal_2k": Workload("bf16_causal_2k", 4, 16, 2048, 2048, 128, True, seed=1002),
    "bf16_causal_8k": Workload("bf16_causal_8k", 2, 32, 8192, 8192, 128, True, amp=2.0, seed=1003),
    "bf16_noncausal_8k": Workload("bf16_noncausal_8k", 2, 32, 8192, 8192, 128, False, amp=2.0,
                                  seed=1003),
    "bf16_varlen_causal": Workload("bf16_varlen_causal", 18, 16, 4096, 4096, 128, True,
                                   seed=1004, varlen=True, n_seqs=16, empty_k_at=(3, 17)),
    "fp8_noncausal_4k": Workload("fp8_noncausal_4k", 4, 16, 4096, 4096, 128, False,
                                 dtype="e4m3", seed=1005),
    "bf16_shortq_longkv": Workload("bf16_shortq_longkv", 1, 8, 128, 65536, 128, False,
                                   seed=1006),
    # grouped-query attention (4 query heads per K/V head) at the 8K causal shape
    "bf16_gqa_causal_8k": Workload("bf16_gqa_causal_8k", 2, 32, 8192, 8192, 128, True, amp=2.0,
                                   seed=1007, heads_k=8),
    # FP8 with one descale per (batch, head) and an E5M2 V
    "fp8_headscale_4k": Workload("fp8_headscale_4k", 4, 16, 4096, 4096, 128, False,
                                 dtype="e4m3", v_dtype="e5m2", descale="head", seed=1008),
    # decoding with a key/value cache: append one token, attend over the filled cache
    "bf16_kvcache_decode": Workload("bf16_kvcache_decode", 16, 32, 1, 8192, 128, True,
                                    seed=1009, heads_k=8, cache_new=1),
}


def quantize_e4m3(x: torch.Tensor):
    """Per-tensor FP8 E4M3 quantisation: descale = amax/448, x8 = rn(x/descale).

    Values are clamped to +-448 before the round-to-nearest cast, which is the
    saturating ("satfinite") reading.  Returns (x8, descale as a python float).
    """
    amax = float(x.abs().max())
    descale = amax / E4M3_MAX if amax > 0 else 1.0
    y = (x / descale).clamp_(-E4M3_MAX, E4M3_MAX)
    return y.to(torch.float8_e4m3fn), descale


def quantize_fp8_per_head(x: torch.Tensor, fmt: str, heads_k: int):
    """FP8 quantisation with one descale per (batch, key/value head).

    x: [B, S, H, D] with H a multiple of heads_k; query heads that share a K/V head
    share a descale (the amax is taken over the whole group).  descale[b, g] =
    amax / max-finite of the format, x8 = rn(clamp(x / descale)).
    Returns (x8, descale fp32 [B, heads_k]).
    """
    dt, mx = _FP8[fmt]
    B, S, H, D = x.shape
    g = x.reshape(B, S, heads_k, H // heads_k, D)
    amax = (g.abs().amax(dim=(1, 3, 4)) if g.numel() else     # [B, heads_k]
            torch.zeros((B, heads_k), dtype=x.dtype))
    descale = torch.where(amax > 0, amax / mx, torch.ones_like(amax)).to(torch.float32)
    y = (g / descale.view(B, 1, heads_k, 1, 1)).clamp_(-mx, mx).reshape(B, S, H, D)
    return y.to(dt), descale


def varlen_lengths(w: Workload, gen: torch.Generator):
    """Per-sequence (seqlen_q, seqlen_k): n_seqs lengths U{1..4096} with Sq = Sk,
    plus len(empty_k_at) sequences with Sq ~ U{1..4096} and Sk = 0, inserted at the
    packed positions empty_k_at (draw order: the n_seqs lengths, then the empty ones)."""
    n_total = w.n_seqs + len(w.empty_k_at)
    draws = torch.randint(1, w.seqlen_q + 1, (n_total,), generator=gen).tolist()
    regular = iter(draws[:w.n_seqs])
    empties = iter(draws[w.n_seqs:])
    sq, sk = [], []
    for pos in range(n_total):
        if pos in w.empty_k_at:
            sq.append(next(empties))
            sk.append(0)
        else:
            s = next(regular)
            sq.append(s)
            sk.append(s)
    return sq, sk


def make_inputs(w: Workload, *, seed: Optional[int] = None, shapes_only_q: Optional[int] = None):
    """Draw (on the CPU) the inputs of a workload.

    Returns a dict with q, k, v (bf16 or float8, CPU; for cache workloads k and v
    are the caches [B, capacity, Hk, D]), descale (q, k, v: python floats, or fp32
    [B, Hk] tensors for per-head descales), k_new / v_new / cache_seqlens (cache
    workloads; drawn after Q, K, V),
    cu_seqlens_q/k (int32 CPU tensors or None), max_seqlen_q/k, seqlens.
    Draw order: Q, K, V (fp32 N(0,1), times amp), then varlen lengths.
    For varlen, the lengths are drawn first from their own generator stream
    (seed + 7919) so that Q/K/V sizes are known before the value draws.
    """
    seed = w.seed if seed is None else seed
    gen = torch.Generator(device="cpu").manual_seed(seed)
    cu_q = cu_k = None
    seqlens = None
    if w.varlen:
        lgen = torch.Generator(device="cpu").manual_seed(seed + 7919)
        sq, sk = varlen_lengths(w, lgen)
        seqlens = (sq, sk)
        cu_q = torch.tensor([0] + list(_cumsum(sq)), dtype=torch.int32)
        cu_k = torch.tensor([0] + list(_cumsum(sk)), dtype=torch.int32)
        q_shape = (int(cu_q[-1]), w.heads, w.head_dim)
        k_shape = (int(cu_k[-1]), w.kv_heads, w.head_dim)
        max_q, max_k = max(sq), max(sk)
    else:
        q_shape = (w.batch, w.seqlen_q, w.heads, w.head_dim)
        k_shape = (w.batch, w.seqlen_k, w.kv_heads, w.head_dim)
        max_q, max_k = w.seqlen_q, w.seqlen_k
    q = torch.randn(q_shape, generator=gen, dtype=torch.float32)
    k = torch.randn(k_shape, generator=gen, dtype=torch.float32)
    v = torch.randn(k_shape, generator=gen, dtype=torch.float32)
    cache = {}
    if w.cache_new:
        # new rows, then the filled length of each sequence's cache (rows past it are
        # random too: they must be ignored)
        nshape = (w.batch, w.cache_new, w.kv_heads, w.head_dim)
        cache["k_new"] = torch.randn(nshape, generator=gen, dtype=torch.float32) * w.amp
        cache["v_new"] = torch.randn(nshape, generator=gen, dtype=torch.float32) * w.amp
        lo = w.seqlen_k // 2
        cache["cache_seqlens"] = torch.randint(lo, w.seqlen_k - w.cache_new + 1, (w.batch,),
                                               generator=gen, dtype=torch.int32)
        if w.dtype != "bf16":
            raise ValueError("cache workloads are drawn in bf16")
        cache["k_new"] = cache["k_new"].to(torch.bfloat16)
        cache["v_new"] = cache["v_new"].to(torch.bfloat16)
    if w.amp != 1.0:
        q.mul_(w.amp)
        k.mul_(w.amp)
        v.mul_(w.amp)
    if w.dtype == "e4m3" and w.descale == "head":
        if w.varlen:
            raise ValueError("per-head descales are drawn for fixed-length workloads only")
        q, dq = quantize_fp8_per_head(q, "e4m3", w.kv_heads)
        k, dk = quantize_fp8_per_head(k, "e4m3", w.kv_heads)
        v, dv = quantize_fp8_per_head(v, w.v_dtype or "e4m3", w.kv_heads)
        descale = (dq, dk, dv)
    elif w.dtype == "e4m3":
        if w.v_dtype not in ("", "e4m3"):
            raise ValueError("a per-tensor E5M2 V is not drawn; use descale='head'")
        q8, dq = quantize_e4m3(q)
        k8, dk = quantize_e4m3(k)
        v8, dv = quantize_e4m3(v)
        q, k, v, descale = q8, k8, v8, (dq, dk, dv)
    else:
        q, k, v = q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)
        descale = (1.0, 1.0, 1.0)
    return dict(q=q, k=k, v=v, descale=descale, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
                max_seqlen_q=max_q, max_seqlen_k=max_k, seqlens=seqlens, **cache)


def make_random(batch, heads, seqlen_q, seqlen_k, head_dim, *, seed, amp=1.0,
                dtype="bf16", heads_k=0, v_dtype="", descale="tensor"):
    """Fixed-length N(0,1)*amp inputs of an arbitrary shape (for edge cases)."""
    w = Workload("custom", batch, heads, seqlen_q, seqlen_k, head_dim, False, dtype=dtype,
                 amp=amp, seed=seed, heads_k=heads_k, v_dtype=v_dtype, descale=descale)
    return make_inputs(w)


def make_varlen(seqlens_q, seqlens_k, heads, head_dim, *, seed, amp=1.0, heads_k=0):
    """Packed varlen bf16 inputs for given per-sequence lengths."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    cu_q = torch.tensor([0] + list(_cumsum(seqlens_q)), dtype=torch.int32)
    cu_k = torch.tensor([0] + list(_cumsum(seqlens_k)), dtype=torch.int32)
    hk = heads_k or heads
    q = torch.randn((int(cu_q[-1]), heads, head_dim), generator=gen) * amp
    k = torch.randn((int(cu_k[-1]), hk, head_dim), generator=gen) * amp
    v = torch.randn((int(cu_k[-1]), hk, head_dim), generator=gen) * amp
    return dict(q=q.to(torch.bfloat16), k=k.to(torch.bfloat16), v=v.to(torch.bfloat16),
                descale=(1.0, 1.0, 1.0), cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
                max_seqlen_q=max(seqlens_q) if seqlens_q else 0,
                max_seqlen_k=max(seqlens_k) if seqlens_k else 0,
                seqlens=(list(seqlens_q), list(seqlens_k)))


def _cumsum(xs):
    t = 0
    for x in xs:
        t += x
        yield t
