"""The exp2-on-FMA-pipe option (CPU): its constants come from the committed
derivation, and the kernel's float32 steps (clamp, round-by-magic-add, degree-3
minimax on the fraction, exponent-field add) stay within the polynomial's error bound
of exp2 over every input the softmax can produce (x = s*scale_log2 - m <= 16)."""
import os
import re

import numpy as np

from exact_attention_forward_gb300 import exp2_poly

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KERNEL = os.path.join(ROOT, "exact_attention_forward_gb300", "csrc", "fa_fwd_kernel.cuh")


def kernel_constants():
    text = open(KERNEL).read()
    c = [float(re.search(rf"kExp2C{i} = ([0-9.eE+-]+)f;", text).group(1)) for i in range(4)]
    magic = float(re.search(r"kRoundMagic = ([0-9.]+)f;", text).group(1))
    return np.array(c, dtype=np.float32), np.float32(magic)


def test_constants_match_the_derivation():
    c, err = exp2_poly.derive()
    kc, magic = kernel_constants()
    assert np.array_equal(kc, c.astype(np.float32))
    assert err < 8e-5
    assert magic == np.float32(1.5 * 2 ** 23)


def emulate(x):
    """The kernel's steps in float32 (f32x2 arithmetic is plain fp32 per lane)."""
    c, magic = kernel_constants()
    x = np.maximum(x.astype(np.float32), np.float32(-125.0))
    r = (x + magic).astype(np.float32)
    f = (x - (r - magic).astype(np.float32)).astype(np.float32)
    p = (c[3] * f + c[2]).astype(np.float32)        # fma rounding differs by <= 1 ulp per step
    p = (p * f + c[1]).astype(np.float32)
    p = (p * f + c[0]).astype(np.float32)
    bits = p.view(np.uint32) + (r.view(np.uint32) << np.uint32(23))
    return bits.astype(np.uint32).view(np.float32)


def test_emulation_error_over_the_softmax_range():
    x = np.concatenate([np.linspace(-125.0, 16.0, 2_000_001, dtype=np.float64),
                        np.arange(-125, 17, dtype=np.float64) + 0.5])
    got = emulate(x).astype(np.float64)
    want = np.exp2(np.maximum(x, -125.0))
    rel = np.abs(got / want - 1.0)
    assert rel.max() < 1e-4, rel.max()
    # and exactly representable powers of two come out (nearly) exact
    xi = np.arange(-120, 17, dtype=np.float64)
    assert np.allclose(emulate(xi), np.exp2(xi), rtol=2e-4)
