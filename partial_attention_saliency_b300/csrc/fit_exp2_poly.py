"""Coefficients of the FMA-pipe 2^f polynomial used by the kernels (exp2_poly2).

The kernels split 2^x = 2^n * 2^f with n = round(x) and f in [-1/2, 1/2]
(Cody and Waite's argument reduction), and evaluate 2^f as a degree-4
polynomial in Horner form.  The polynomial minimises the maximum RELATIVE
error on [-1/2, 1/2]; it is found here by Lawson's iteratively reweighted
least squares (each pass re-weights every sample point by its current
absolute error, which converges to the minimax fit) on a Chebyshev grid, and
the float64 result is rounded to float32.

    python -m partial_attention_saliency_b300.csrc.fit_exp2_poly
        (or python partial_attention_saliency_b300/csrc/fit_exp2_poly.py)

prints the coefficients, highest degree first, as C hexadecimal float
literals, and the maximum relative error of the float32 polynomial
evaluated in float64.  The constants in common.cuh are this script's output.
"""
from __future__ import annotations

import numpy as np

DEGREE = 4
GRID = 40001
PASSES = 2000


def fit(degree: int = DEGREE, grid: int = GRID, passes: int = PASSES):
    """Returns (float32 coefficients, lowest degree first; max relative error
    of the float32 polynomial on the grid, evaluated in float64)."""
    f = np.cos(np.linspace(0.0, np.pi, grid))[::-1] * 0.5
    y = np.exp2(f)
    V = np.vander(f, degree + 1, increasing=True)
    w = np.full(grid, 1.0 / grid)
    c = None
    for _ in range(passes):
        sw = np.sqrt(w)
        c, *_ = np.linalg.lstsq(V / y[:, None] * sw[:, None], sw, rcond=None)
        e = (V @ c) / y - 1.0
        w = w * np.abs(e)
        w /= w.sum()
    c32 = c.astype(np.float32)
    err = float(np.max(np.abs((V @ c32.astype(np.float64)) / y - 1.0)))
    return c32, err


def c_literal(v: np.float32) -> str:
    m, e = float(v).hex().split("p")
    return m.rstrip("0") + "p" + e + "f"


if __name__ == "__main__":
    c32, err = fit()
    print("coefficients, highest degree first:", ", ".join(c_literal(v) for v in c32[::-1]))
    print(f"max relative error of the float32 polynomial on [-1/2, 1/2]: {err:.4g}")
