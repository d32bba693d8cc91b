"""Coefficients of the polynomial 2^f the prefill's softmax evaluates on the
FMA pipe for part of each row's exponentials (csrc/common.cuh, ex2_poly2).

Method: 2^x = 2^j * 2^f with j = rint(x) and |f| <= 1/2 (the Cody-Waite
range reduction, exact in binary floating point), and 2^f approximated by
p(f) = 1 + a1 f + a2 f^2 + a3 f^3 + a4 f^4 whose maximum relative error
over [-1/2, 1/2] is minimised (a Chebyshev / minimax fit, computed here as a
linear program over a dense grid: minimise t subject to
-t <= p(f_i) / 2^f_i - 1 <= t).  The constant term is fixed at exactly 1 so
that p(0) = 1: x = 0 (the row's maximum) gives exactly 1, and x clamped to
-127 gives exactly +0.

    python -m exact_io_aware_106_b300.exp2_poly     # prints the fp32 coefficients

The printed values are the ones written into common.cuh; tests/test_exp2_poly.py
checks the committed constants' fp32 error bound on the CPU.
"""
from __future__ import annotations

import numpy as np

DEGREE = 4


def fit(degree: int = DEGREE, grid: int = 4001):
    """Minimax relative-error fit of 2^f on [-1/2, 1/2] with p(0) = 1;
    returns (a_1 .. a_degree as float64, max relative error on the grid)."""
    from scipy.optimize import linprog

    f = np.linspace(-0.5, 0.5, grid)
    ex = 2.0 ** f
    A = np.stack([f ** k / ex for k in range(1, degree + 1)], axis=1)
    b0 = 1.0 / ex - 1.0                      # relative error = A a + b0
    nv = degree + 1
    c = np.zeros(nv)
    c[-1] = 1.0                              # minimise t
    ones = np.ones((grid, 1))
    A_ub = np.vstack([np.hstack([A, -ones]), np.hstack([-A, -ones])])
    b_ub = np.concatenate([-b0, b0])
    r = linprog(c, A_ub=A_ub, b_ub=b_ub, bounds=[(None, None)] * nv, method="highs")
    if not r.success:
        raise RuntimeError(r.message)
    return r.x[:degree], float(r.x[-1])


def eval_fp32(coef, x):
    """The kernel's evaluation simulated in fp32 (round to nearest after every
    operation; fma rounded once): clamp, rint by the 1.5 * 2^23 addition,
    Horner, and the exponent added to the bits."""
    x = np.maximum(np.asarray(x, np.float32), np.float32(-127.0))
    magic = np.float32(12582912.0)
    t = (x + magic).astype(np.float32)
    f = (x - (t - magic).astype(np.float32)).astype(np.float32)
    a = [np.float32(v) for v in coef]
    # fma: the exact product of two fp32 values plus the addend, rounded once
    # (extended precision holds the sum, so only the final rounding is seen)
    fd = f.astype(np.longdouble)
    p = np.full(f.shape, a[-1], np.float32)
    for k in range(len(a) - 2, -1, -1):
        p = (p.astype(np.longdouble) * fd + np.longdouble(a[k])).astype(np.float32)
    p = (p.astype(np.longdouble) * fd + np.longdouble(1.0)).astype(np.float32)
    bits = p.view(np.uint32).astype(np.uint64) + (t.view(np.uint32).astype(np.uint64) << 23)
    return (bits & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


if __name__ == "__main__":
    a, err = fit()
    print(f"degree {DEGREE}, minimax relative error {err:.3e}")
    for k, v in enumerate(a, 1):
        print(f"a{k} = {np.float32(v)!r}  ({float(np.float32(v)).hex()})")
