"""Shared helpers of the GPU parity tests: run the CUDA path into outputs
pre-filled with NaN, compute the oracle over whole workloads (cached per
session, so several tests share one fp64 pass), and compare element by element
with the tolerances of the method: max|dO| <= 2e-2 for bf16 inputs, 6e-2 for
e4m3 inputs, |dLSE| <= 1e-3 over finite LSE; -inf LSE and zero O must match
exactly, and every other output element must have been written (finite).

Two error terms of bf16 arithmetic are added to the O bound, each only where
it can exceed the tolerance, and each derived rather than fitted:

* Output rounding.  O is stored in bf16; rounding the kernel's fp32 result to
  the nearest bf16 value moves it by up to half an ulp of that value, 2^-5 =
  0.031 for |O| in [8, 16) -- more than 2e-2 by itself.  Where the largest
  half-ulp of the oracle's O (rounded to bf16) exceeds the tolerance (the
  x2-amplitude 8K workloads), the bound per element is tol + half_ulp(O_ref).
* Rounding of P.  The kernel feeds P = 2^(s*scale_log2 - m) to the PV
  product as bf16 (relative error <= 2^-9, round to nearest) while the
  normaliser l sums the unrounded fp32 values, so each O element moves by at
  most 2^-9 * sum_j w_j |v_jd| (w = the softmax weights), i.e. 2^-9 times
  the oracle's output over |V|.  Elements still past the bound above get this
  term, computed exactly for their rows by the oracle over |V|; the records
  count them.
"""
import functools

import numpy as np
import torch

import oracle
import exact_attention_forward_gb300 as fa

TOL_O = {"bf16": 2e-2, "e4m3": 6e-2}
TOL_LSE = 1e-3

# (what, dtype, max|dO|, max|dLSE|, max|O_ref|, bound, rows compared) of every comparison
# this session; printed at the end of the run by conftest.py
RECORDS = []


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 values at the bf16 value nearest x (0 at 0): bf16 keeps 8
    significant bits, so for a nearest value r in [2^e, 2^(e+1)) the half-ulp is 2^(e-8)."""
    r = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    r = r.to(torch.float64).abs().numpy()
    out = np.zeros_like(r)
    nz = r > 0
    out[nz] = np.exp2(np.floor(np.log2(r[nz])) - 8.0)
    return out


def to_dev(x, dev="cuda"):
    out = dict(x)
    for n in ("q", "k", "v"):
        out[n] = x[n].to(dev)
    for n in ("cu_seqlens_q", "cu_seqlens_k"):
        if x.get(n) is not None:
            out[n] = x[n].to(dev)
    return out


def nan_outputs(q, v, lse_shape, dev="cuda"):
    """O and LSE buffers pre-filled with NaN: an element the kernel never writes stays NaN."""
    o = torch.full(tuple(q.shape[:-1]) + (v.shape[-1],), float("nan"), dtype=torch.bfloat16,
                   device=dev)
    lse = torch.full(lse_shape, float("nan"), dtype=torch.float32, device=dev)
    return o, lse


def lse_shape_of(x):
    q = x["q"]
    if x.get("cu_seqlens_q") is not None:
        return (q.shape[1], q.shape[0])
    return (q.shape[0], q.shape[2], q.shape[1])


def run_gpu(x, *, causal, softmax_scale, workspace="auto", cta_pair=False):
    d = to_dev(x)
    o, lse = nan_outputs(d["q"], d["v"], lse_shape_of(x))
    fa.fwd(d["q"], d["k"], d["v"], causal=causal, softmax_scale=softmax_scale,
           cu_seqlens_q=d.get("cu_seqlens_q"), cu_seqlens_k=d.get("cu_seqlens_k"),
           max_seqlen_q=x.get("max_seqlen_q"), max_seqlen_k=x.get("max_seqlen_k"),
           descale=x["descale"] if x["q"].dtype == torch.float8_e4m3fn else None,
           workspace=workspace, cta_pair=cta_pair, out=o, lse=lse)
    torch.cuda.synchronize()
    st, flags = fa.device_error(clear=True)
    assert st == 0, f"device error word {flags:#x}"
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


P_ROUND_REL = 2.0 ** -9  # relative half-ulp of bf16 (8 significant bits), P's type in the PV product


def _row_index(shape_o, flat_rows):
    """Oracle (b, h, i) triples of O rows given as flat indices into O's leading dims."""
    if len(shape_o) == 4:  # [B, Sq, H, D]
        b, i, h = np.unravel_index(flat_rows, shape_o[:3])
        return np.stack([b, h, i], axis=1).astype(np.int64)
    raise ValueError("P-rounding term needs fixed-length O [B, Sq, H, D] or a row mapper")


def compare(o, lse, o_ref, lse_ref, dtype="bf16", what="", o_abs_v=None):
    """Element-wise check; returns (max|dO|, max|dLSE|, max|O_ref|).

    o_abs_v(flat_rows) -> [n, Dv]: the oracle's O over |V| for the given O rows (flat
    indices into O's leading dimensions); enables the bf16 P-rounding term."""
    tol_o = TOL_O[dtype]
    assert o.shape == o_ref.shape and lse.shape == lse_ref.shape
    assert not np.any(np.isnan(o)), f"{what}: {int(np.isnan(o).sum())} O elements never written"
    assert not np.any(np.isnan(lse)), f"{what}: {int(np.isnan(lse).sum())} LSE rows never written"
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse), fin), f"{what}: finite-LSE pattern differs"
    assert np.all(lse[~fin] == -np.inf), f"{what}: LSE must be -inf where no key is visible"
    d_lse = float(np.abs(lse[fin] - lse_ref[fin]).max()) if fin.any() else 0.0
    d_o = np.abs(o - o_ref)
    hu = half_ulp_bf16(o_ref) if o_ref.size else np.zeros(0)
    rounding = bool(hu.size) and float(hu.max()) > tol_o
    excess = d_o - (tol_o + hu if rounding else tol_o)
    bound = f"{tol_o:g}" + (" + half-ulp(O_ref)" if rounding else "")
    n_p = 0
    if excess.size and float(excess.max()) > 0 and o_abs_v is not None and dtype == "bf16":
        rows2 = excess.reshape(-1, excess.shape[-1])
        bad = np.nonzero((rows2 > 0).any(axis=1))[0]
        n_p = int((rows2[bad] > 0).sum())
        ov = np.asarray(o_abs_v(bad), dtype=np.float64).reshape(len(bad), -1)
        rows2[bad] -= P_ROUND_REL * ov
        bound += f" + 2^-9 P|V| on {n_p} elements"
    worst = float(excess.max()) if excess.size else 0.0
    max_do = float(d_o.max()) if d_o.size else 0.0
    max_o = float(np.abs(o_ref).max()) if o_ref.size else 0.0
    RECORDS.append((what, dtype, max_do, d_lse, max_o, bound, int(lse_ref.size)))
    assert worst <= 0, (f"{what}: max|dO| {max_do:.3e} exceeds the bound by {worst:.3e} "
                        f"(max|O_ref| {max_o:.2f}; bound {bound})")
    assert d_lse <= TOL_LSE, f"{what}: max|dLSE| = {d_lse:.3e}"
    # rows where no key is visible: O exactly 0
    if (~fin).any():
        if lse.ndim == 3:  # [B, H, Sq] against O [B, Sq, H, D]
            empty = np.transpose(~fin, (0, 2, 1))
        elif lse.ndim == 2:  # [H, total] against O [total, H, D]
            empty = np.transpose(~fin, (1, 0))
        else:  # gathered rows: [n] against [n, D]
            empty = ~fin
        assert np.all(o[empty] == 0), f"{what}: O must be 0 where no key is visible"
    return max_do, d_lse, max_o


def oracle_abs_v(x, *, softmax_scale, causal):
    """o_abs_v for compare(): the oracle's O over |V| (the softmax weights applied to the
    absolute values) for fixed-length rows given as flat indices into O [B, Sq, H, D]."""
    v_abs = x["v"].abs()  # exact in bf16
    shape = (x["q"].shape[0], x["q"].shape[1], x["q"].shape[2], x["v"].shape[-1])

    def f(flat_rows):
        rows = _row_index(shape, flat_rows)
        return oracle.attention_rows(x["q"], x["k"], v_abs, rows, softmax_scale=softmax_scale,
                                     causal=causal)[0]
    return f


def assert_all_written(o, lse, what=""):
    """Whole-tensor check for tests that compare sampled rows only: nothing left NaN."""
    assert not np.any(np.isnan(o)), f"{what}: {int(np.isnan(o).sum())} O elements never written"
    assert not np.any(np.isnan(lse)), f"{what}: {int(np.isnan(lse).sum())} LSE rows never written"
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"


@functools.lru_cache(maxsize=None)
def workload_inputs(name):
    from exact_attention_forward_gb300 import inputs
    return inputs.make_inputs(inputs.WORKLOADS[name])


@functools.lru_cache(maxsize=None)
def oracle_full(name):
    """The oracle's O and LSE over a whole configured workload (every row), computed once
    per test session and shared by the tests that run that workload."""
    from exact_attention_forward_gb300 import inputs
    w = inputs.WORKLOADS[name]
    x = workload_inputs(name)
    kw = {"descale": x["descale"]} if w.dtype == "e4m3" else {}
    return oracle.attention(x["q"], x["k"], x["v"], softmax_scale=w.softmax_scale,
                            causal=w.causal, cu_seqlens_q=x.get("cu_seqlens_q"),
                            cu_seqlens_k=x.get("cu_seqlens_k"), **kw)


def sample_rows(batch, heads, seqlen_q, n_random, seed, seqlens_q=None):
    """(b, h, i) triples: tile-boundary rows (0, 127, 128, 255, 256, last) of every
    (b, h) plus n_random seeded random rows."""
    rng = np.random.default_rng(seed)
    rows = []
    for b in range(batch):
        sq = seqlen_q if seqlens_q is None else int(seqlens_q[b])
        if sq == 0:
            continue
        special = sorted({i for i in (0, 127, 128, 255, 256, sq // 2, sq - 129, sq - 128, sq - 1)
                          if 0 <= i < sq})
        for h in range(heads):
            rows += [(b, h, i) for i in special]
    bs = rng.integers(0, batch, size=n_random)
    for b in bs:
        sq = seqlen_q if seqlens_q is None else int(seqlens_q[b])
        if sq == 0:
            continue
        rows.append((int(b), int(rng.integers(0, heads)), int(rng.integers(0, sq))))
    return np.array(sorted(set(rows)), dtype=np.int64)


def gather_rows(o, lse, rows, varlen=False, cu_q=None):
    b, h, i = rows[:, 0], rows[:, 1], rows[:, 2]
    if varlen:
        pos = np.asarray(cu_q, dtype=np.int64)[b] + i
        return o[pos, h], lse[h, pos]
    return o[b, i, h], lse[b, h, i]


def e4m3_half_spacing(p: np.ndarray) -> np.ndarray:
    """Half the spacing of e4m3 values around p >= 0 (round to nearest): 3 mantissa bits in
    the normal range [2^-6, 448], spacing 2^-9 below it (subnormals, and values that round
    to zero)."""
    p = np.asarray(p, dtype=np.float64)
    out = np.full(p.shape, 2.0 ** -10)
    nrm = p >= 2.0 ** -6
    out[nrm] = np.exp2(np.floor(np.log2(p[nrm])) - 4.0)
    return out


def fp8_p_bound(w: np.ndarray, v_abs: np.ndarray, lags=np.linspace(0.0, 8.0, 33)) -> np.ndarray:
    """Worst-case change of O from rounding P to e4m3, for rows with softmax weights w [n, Sk]
    over keys with |V| v_abs [Sk, Dv] (or [n, Sk, Dv]): the kernel exponentiates against a
    reference maximum that lags the row's maximum by up to 2^8, so P_j = 2^lag w_j / w_max and
    the normaliser is L = 2^lag / w_max; each P_j moves by at most half an e4m3 spacing, and
    |dO_d| <= sum_j hs(P_j) |v_jd| / L.  Returns the largest bound over the lags, [n, Dv]."""
    w = np.asarray(w, dtype=np.float64)
    wmax = np.maximum(w.max(axis=1, keepdims=True), 1e-300)
    best = None
    for lag in lags:
        p = np.exp2(lag) * w / wmax
        hs = np.where(w > 0, e4m3_half_spacing(p), 0.0) * wmax / np.exp2(lag)
        b = np.einsum("nk,nkd->nd", hs, v_abs) if v_abs.ndim == 3 else hs @ v_abs
        best = b if best is None else np.maximum(best, b)
    return best
