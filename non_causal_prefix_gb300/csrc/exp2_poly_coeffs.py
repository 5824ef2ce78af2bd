"""Coefficients of the polynomial exp2 used for part of the softmax exponentials.

The kernels split x = j + f with j = round(x) (an integer, put into the float's
exponent field) and f in [-1/2, 1/2], then approximate 2^f by
p(f) = 1 + c1 f + c2 f^2 + c3 f^3 (Horner form, fp32 FMAs).  This is the
classic Cody-Waite style range reduction followed by a minimax polynomial on
the reduced range.  The constant term is pinned to 1 so that p(0) = 1 exactly:
integer x give exact powers of two and x = -127 (the clamp) gives exactly +0.

c1..c3 minimise max |p(f) / 2^f - 1| over a dense grid of [-1/2, 1/2], solved
as a linear programme.  The maximum relative error is about 1.0e-4, twenty
times below the half-ulp of bf16 (2^-9), the precision the probabilities are
rounded to before the P V product.

Run this file to print the coefficients as fp32 hex literals; the test suite
checks that the CUDA source uses these values.
"""
from __future__ import annotations

import numpy as np


def solve(grid_points: int = 4001):
    from scipy.optimize import linprog
    g = np.linspace(-0.5, 0.5, grid_points)
    w = 2.0 ** g
    a = np.stack([g / w, g ** 2 / w, g ** 3 / w], 1)
    b0 = 1.0 / w - 1.0
    ones = np.ones((g.size, 1))
    a_ub = np.vstack([np.hstack([a, -ones]), np.hstack([-a, -ones])])
    b_ub = np.concatenate([-b0, b0])
    res = linprog(np.array([0.0, 0.0, 0.0, 1.0]), A_ub=a_ub, b_ub=b_ub,
                  bounds=[(None, None)] * 4, method="highs")
    if not res.success:
        raise RuntimeError(res.message)
    return [float(np.float32(c)) for c in res.x[:3]], float(res.x[3])


def max_rel_error_fp32(coeffs, n: int = 1_000_001) -> float:
    """Max relative error of p evaluated in fp32 (Horner) over [-1/2, 1/2]."""
    f = np.linspace(-0.5, 0.5, n).astype(np.float32)
    c1, c2, c3 = (np.float32(c) for c in coeffs)
    p = np.float32(1) + f * (c1 + f * (c2 + f * c3))
    return float(np.abs(p.astype(np.float64) / 2.0 ** f.astype(np.float64) - 1).max())


if __name__ == "__main__":
    coeffs, err = solve()
    for name, c in zip(("C1", "C2", "C3"), coeffs):
        print(f"{name} = {c.hex()}  ({c!r})")
    print(f"minimax relative error {err:.3e}; fp32 evaluation {max_rel_error_fp32(coeffs):.3e}")
