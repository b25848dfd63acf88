"""Derives the polynomial used by the kernel's software 2^x.

Method: Remez exchange for the minimax *relative* error of a degree-n
polynomial P(f) ~ 2^f on f in [-1/2, 1/2] (the reduced argument after
rounding x to the nearest integer, x = k + f).  The weight is 1 / 2^f, so the
alternation conditions are P(x_i) - 2^(x_i) = (-1)^i * E * 2^(x_i).  All
arithmetic is float64; the printed coefficients are then rounded to float32
and the error of the float32 polynomial evaluated in float32 Horner form is
reported, which is the number the kernel's tests check against.

    python gen_exp2_poly.py [degree]
"""
from __future__ import annotations

import sys

import numpy as np


def remez_exp2(degree: int, lo: float = -0.5, hi: float = 0.5, iters: int = 30):
    n = degree
    # Chebyshev extrema as the initial reference (n + 2 points).
    k = np.arange(n + 2)
    x = 0.5 * (lo + hi) + 0.5 * (hi - lo) * np.cos(np.pi * k[::-1] / (n + 1))
    grid = np.linspace(lo, hi, 200001)
    coef, E = None, None
    for _ in range(iters):
        # Solve sum_j c_j x_i^j - (-1)^i E 2^x_i = 2^x_i for c_0..c_n, E.
        A = np.zeros((n + 2, n + 2))
        for j in range(n + 1):
            A[:, j] = x ** j
        A[:, n + 1] = -((-1.0) ** np.arange(n + 2)) * np.exp2(x)
        sol = np.linalg.solve(A, np.exp2(x))
        coef, E = sol[: n + 1], sol[n + 1]
        err = (np.polyval(coef[::-1], grid) - np.exp2(grid)) / np.exp2(grid)
        # New reference: the n + 2 alternating extrema of the error.
        sign = np.sign(err)
        idx = np.flatnonzero(np.diff(sign) != 0)
        segments = np.split(np.arange(grid.size), idx + 1)
        ext = [seg[np.argmax(np.abs(err[seg]))] for seg in segments]
        if len(ext) != n + 2:
            break
        x_new = grid[ext]
        if np.allclose(x_new, x, atol=1e-12, rtol=0):
            break
        x = x_new
    return coef, abs(E)


def float32_error(coef32, lo=-0.5, hi=0.5):
    f = np.linspace(lo, hi, 400001).astype(np.float32)
    p = np.full_like(f, coef32[-1])
    for c in coef32[-2::-1]:
        p = (p * f + c).astype(np.float32)
    exact = np.exp2(f.astype(np.float64))
    return float(np.max(np.abs(p.astype(np.float64) - exact) / exact))


if __name__ == "__main__":
    deg = int(sys.argv[1]) if len(sys.argv) > 1 else 3
    c, e = remez_exp2(deg)
    c32 = np.asarray(c, dtype=np.float32)
    print("degree %d, minimax relative error (float64) %.3e, float32 Horner %.3e" % (deg, e, float32_error(c32)))
    for i, v in enumerate(c32):
        print("  c%d = %s  (%.9e)" % (i, float(v).hex(), float(v)))
