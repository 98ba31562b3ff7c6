"""Fit the FMA-pipe polynomial for 2^f, f in [-1/2, 1/2], used by the kernels.

The FA4 design computes part of the softmax exponentials with a polynomial on
the FMA pipe instead of the exponential unit ("FlashAttention" wiki note, FA4
item (2): software-emulated exp by polynomial approximation).  The pages give
no degree or coefficients, so they are fitted here, from the mathematics only:

    2^x = 2^j * 2^f,   j = round(x),  f = x - j in [-1/2, 1/2]
    2^f ~ p(f) = 1 + f*(c1 + f*(c2 + f*c3))

p(0) = 1 exactly (so a row's maximum element maps to exactly 1), and c1..c3
minimise the maximum relative error max |p(f) - 2^f| / 2^f on a dense grid,
posed as a linear program (Chebyshev approximation).  Run this file to print
the coefficients; the kernels carry them as literals and a test checks that
the two agree and that the evaluation error stays below 1e-4.
"""
from __future__ import annotations

import numpy as np


def fit(n_grid: int = 4001):
    from scipy.optimize import linprog

    f = np.linspace(-0.5, 0.5, n_grid)
    t = np.exp2(f)
    # variables: c1, c2, c3, E ; minimise E
    # |1 + c1 f + c2 f^2 + c3 f^3 - t| <= E t
    basis = np.stack([f, f * f, f * f * f], axis=1)
    a_up = np.hstack([basis, -t[:, None]])      #  (1 + B c - t) <= E t
    a_dn = np.hstack([-basis, -t[:, None]])     # -(1 + B c - t) <= E t
    b_up = t - 1.0
    b_dn = 1.0 - t
    res = linprog(c=[0, 0, 0, 1], A_ub=np.vstack([a_up, a_dn]), b_ub=np.concatenate([b_up, b_dn]),
                  bounds=[(None, None)] * 3 + [(0, None)], method="highs")
    assert res.success, res.message
    c1, c2, c3, err = res.x
    return (float(c1), float(c2), float(c3)), float(err)


if __name__ == "__main__":
    (c1, c2, c3), err = fit()
    print("c1 = %.9e\nc2 = %.9e\nc3 = %.9e\nmax relative error = %.3e" % (c1, c2, c3, err))
