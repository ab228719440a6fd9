"""CPU: the error model of P rounded to e4m3 (the FP8 path) against an emulation of the
kernel's arithmetic.  The forward kernel exponentiates against a reference maximum that
lags the row's true maximum by up to 2^8 (lazy rescaling), rounds P to e4m3 for the PV
product, sums the unrounded fp32 P into the normaliser l, and stores O = v_descale (P_e4m3
V) / l.  Emulated in numpy with torch's e4m3 rounding, every element must stay within
fp8_p_bound (plus the bf16 rounding of the output), for lags across [0, 8] and for value
spreads up to 1.5 N(0,1), and the bound must not be vacuous (far above the error)."""
import numpy as np
import torch

from parity_util import e4m3_half_spacing, fp8_p_bound, half_ulp_bf16


def _e4m3(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).to(
        torch.float64).numpy()


def _bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).to(
        torch.float64).numpy()


def test_half_spacing_matches_the_format():
    # e4m3 values are exactly representable: a value one half-spacing above rounds back
    for p in (2.0 ** -9, 2.0 ** -7, 2.0 ** -6, 0.5, 1.0, 1.125, 3.0, 96.0, 240.0):
        hs = float(e4m3_half_spacing(np.array([p]))[0])
        assert _e4m3([p])[0] == p
        assert _e4m3([p + 0.99 * hs])[0] == p and _e4m3([p + 1.01 * hs])[0] > p


def test_bound_holds_for_lagging_maxima_and_wide_spreads():
    rng = np.random.default_rng(3)
    sq, sk, d = 48, 300, 64
    ratios = []
    for amp in (1.0, 1.5):
        q = _e4m3(rng.normal(size=(sq, d)) * amp)
        k = _e4m3(rng.normal(size=(sk, d)) * amp)
        v = _e4m3(rng.normal(size=(sk, d)) * amp)
        s = (q @ k.T) * d ** -0.5
        w = np.exp(s - s.max(axis=1, keepdims=True))
        w /= w.sum(axis=1, keepdims=True)
        o_ref = w @ v
        bound = fp8_p_bound(w, np.abs(v)) + half_ulp_bf16(o_ref) + 1e-6
        for lag in (0.0, 0.3, 2.7, 5.0, 7.99):
            x = (s - s.max(axis=1, keepdims=True)) * np.log2(np.e) + lag
            p = np.exp2(x)
            o = _bf16((_e4m3(p) @ v) / p.sum(axis=1, keepdims=True))
            err = np.abs(o - o_ref)
            assert np.all(err <= bound), (amp, lag, float((err - bound).max()))
            ratios.append(float(err.max() / bound.max()))
    assert max(ratios) > 0.1  # the bound is a useful one, not orders of magnitude loose
