"""Derivation of the polynomial used for exp2 on the FMA pipe.

2^x = 2^n * 2^f with n = round(x), f = x - n in [-1/2, 1/2] (Cody-Waite style range
reduction); 2^f is approximated by a degree-3 polynomial whose maximum *relative*
error on [-1/2, 1/2] is minimised (minimax), found here by linear programming over a
dense Chebyshev-spaced grid.  The kernel (csrc/fa_fwd_kernel.cuh, kExp2C0..C3) holds
the float32 roundings of these coefficients; tests/test_exp2_poly.py re-derives them
and checks the kernel's arithmetic against exp2.

    python -m exact_attention_forward_gb300.exp2_poly
"""
from __future__ import annotations

import numpy as np


def derive(degree: int = 3, n_grid: int = 4001):
    """Coefficients c0..c_degree (float64) and the max relative error on [-1/2, 1/2]."""
    from scipy.optimize import linprog

    f = np.cos(np.linspace(0.0, np.pi, n_grid)) * 0.5
    y = np.exp2(f)
    a = np.vander(f, degree + 1, increasing=True)
    # minimise t subject to |a c - y| <= t y
    a_ub = np.vstack([np.hstack([a, -y[:, None]]), np.hstack([-a, -y[:, None]])])
    b_ub = np.concatenate([y, -y])
    cost = np.zeros(degree + 2)
    cost[-1] = 1.0
    res = linprog(cost, A_ub=a_ub, b_ub=b_ub,
                  bounds=[(None, None)] * (degree + 1) + [(0, None)], method="highs")
    if not res.success:
        raise RuntimeError(res.message)
    c = res.x[:-1]
    ff = np.linspace(-0.5, 0.5, 200001)
    err = float(np.abs(np.polyval(c[::-1], ff) / np.exp2(ff) - 1.0).max())
    return c, err


if __name__ == "__main__":
    c, err = derive()
    print("coefficients (float32):", [repr(float(np.float32(x))) for x in c])
    print("max relative error:", err)
