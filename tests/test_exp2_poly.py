"""The FMA-pipe polynomial exp2 used by the forward's exponential split.

The pages ask for part of the softmax exponentials to be computed by a
polynomial on the FMA pipe ("FlashAttention" wiki note, FA4 item (2)) but give
no polynomial.  exact_attention_49_gb300/fit_exp2.py fits one; the kernels
carry its coefficients as literals.  These host-only tests check that the
literals are the fit's output, and emulate the kernel's steps in float32
(clamp, round-to-integer by adding 1.5*2^23, Horner, add j into the exponent
field) against numpy's float64 exp2 over the whole range the softmax uses.
"""
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "exact_attention_49_gb300", "csrc", "sm103.cuh")


def kernel_coefficients():
    text = open(HEADER).read()
    return tuple(float(re.search(r"kExp2C%d = ([0-9.eE+-]+)f;" % k, text).group(1)) for k in (1, 2, 3))


def emulate(x, c1, c2, c3):
    """The kernel's ex2_poly2, elementwise, in float32 arithmetic."""
    f32 = np.float32
    x = np.maximum(x.astype(f32), f32(-127.0))
    magic = f32(12582912.0)
    t = (x + magic).astype(f32)
    j = (t - magic).astype(f32)
    f = (x - j).astype(f32)
    # Horner with fused multiply-adds: evaluate each step in float64 and round once
    q = (np.float64(c3) * f + np.float64(c2)).astype(f32)
    q = (q.astype(np.float64) * f + np.float64(c1)).astype(f32)
    q = (q.astype(np.float64) * f + 1.0).astype(f32)
    bits = q.view(np.uint32).astype(np.uint64) + (t.view(np.uint32).astype(np.uint64) << np.uint64(23))
    return (bits & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.float32)


def test_literals_match_the_fit():
    pytest.importorskip("scipy")
    from exact_attention_49_gb300.fit_exp2 import fit
    (c1, c2, c3), err = fit()
    k1, k2, k3 = kernel_coefficients()
    np.testing.assert_allclose([k1, k2, k3], [c1, c2, c3], rtol=1e-8)
    assert err < 1.1e-4


def test_relative_error_over_the_softmax_range():
    c1, c2, c3 = kernel_coefficients()
    x = np.linspace(-126.0, 0.0, 2_000_001).astype(np.float32)
    got = emulate(x, c1, c2, c3).astype(np.float64)
    want = np.exp2(x.astype(np.float64))
    rel = np.abs(got - want) / want
    assert rel.max() < 2e-4, rel.max()


def test_special_values():
    c1, c2, c3 = kernel_coefficients()
    x = np.array([0.0, -np.inf, -200.0, -127.0, -1.0, -0.5, -8.0], np.float32)
    y = emulate(x, c1, c2, c3)
    assert y[0] == 1.0                     # the row maximum maps to exactly 1
    assert y[1] == 0.0 and y[2] == 0.0     # masked entries contribute exactly 0
    assert y[3] == 0.0
    np.testing.assert_allclose(y[4:], np.exp2(x[4:].astype(np.float64)), rtol=2e-4)
    # never negative, never NaN, monotone enough to keep the row max the largest p
    z = emulate(np.linspace(-127.0, 0.0, 100001).astype(np.float32), c1, c2, c3)
    assert np.all(z >= 0) and np.all(np.isfinite(z))
