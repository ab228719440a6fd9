"""CPU: the O bound of the GPU parity tests against an emulation of the kernel's
arithmetic.  The forward kernel exponentiates against a reference maximum m that
may lag the row's true maximum (lazy rescaling: p = 2^(s*scale_log2 - m) up to
2^16 for bf16 P), rounds P to bf16 for the PV product, sums the unrounded fp32 P
into the normaliser l, and stores O = (P_bf16 V) / l in bf16.  Emulated here in
numpy on rows that one key dominates (the case that makes the P-rounding error
systematic), the bound tol + half_ulp(O_ref) + 2^-9 (P|V|) must hold for every
element and every lag, and the P term must be needed for large |V|."""
import numpy as np
import torch

import oracle
from parity_util import P_ROUND_REL, TOL_O, half_ulp_bf16


def _bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).to(
        torch.float64).numpy()


def _emulate(q, k, v, scale, lag):
    """Kernel arithmetic for one (batch, head): fp64 stand-in for fp32, bf16 P and O."""
    s = (q @ k.T) * scale * np.log2(np.e)  # scores in log2 units
    m = s.max(axis=1, keepdims=True) - lag  # the lagging reference maximum
    p = np.exp2(s - m)
    o = (_bf16(p) @ v) / p.sum(axis=1, keepdims=True)
    return _bf16(o)


def test_bound_holds_with_the_p_term_and_needs_it():
    rng = np.random.default_rng(0)
    sq, sk, d = 64, 200, 32
    scale = d ** -0.5
    needed = False
    for amp in (1.0, 4.0, 12.0):
        q = _bf16(rng.normal(size=(sq, d)) * 3.0)
        k = _bf16(rng.normal(size=(sk, d)) * 3.0)  # peaked softmax: one key dominates
        v = _bf16(rng.normal(size=(sk, d)) * amp)
        qt, kt, vt = (torch.from_numpy(a[None, :, None, :]).to(torch.bfloat16) for a in (q, k, v))
        o_ref, _ = oracle.attention(qt, kt, vt, softmax_scale=scale)
        o_abs, _ = oracle.attention(qt, kt, vt.abs(), softmax_scale=scale)
        o_ref, o_abs = o_ref[0, :, 0], o_abs[0, :, 0]
        for lag in (0.0, 0.37, 5.5, 15.9):
            o = _emulate(q, k, v, scale, lag)
            d_o = np.abs(o - o_ref)
            bound = TOL_O["bf16"] + half_ulp_bf16(o_ref) + P_ROUND_REL * o_abs
            assert np.all(d_o <= bound), (amp, lag, float((d_o - bound).max()))
            if np.any(d_o > TOL_O["bf16"] + half_ulp_bf16(o_ref)):
                needed = True
    assert needed  # at |V| ~ 12 the P-rounding term is what keeps the bound
