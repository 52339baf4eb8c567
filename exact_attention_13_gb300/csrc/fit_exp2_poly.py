"""Fit the polynomial the softmax uses to emulate 2^f on [0, 1) with FMAs.

"FlashAttention4 精读", section 3.1.3 "Emulation of the exponential function": split
x = n + f (n = floor(x), f in [0, 1)), compute 2^f by a low-degree polynomial whose constant
term is 1, in Horner form, and add n to the exponent field.  The page's coefficients came from a
minimax fit of the relative error and are not printed, so this script makes its own: a Remez
exchange for

    p(f) = 1 + a1 f + a2 f^2 + a3 f^3,   minimising  max_{f in [0,1]} |p(f) / 2^f - 1|

in fp64, then rounds the coefficients to fp32 and reports the error of the rounded polynomial
evaluated in fp32 Horner form (fma) on a dense grid.  The page's figure for degree 3 is a maximum
relative error of 8.77e-5.

Run: python fit_exp2_poly.py   (prints the coefficients as C float literals)
"""
from __future__ import annotations

import numpy as np


def remez(degree: int = 3, iters: int = 40):
    # unknowns a1..a_deg and the levelled error E; constraint p(0) = 1 is built in
    k = degree + 1  # number of alternation points
    x = 0.5 - 0.5 * np.cos(np.pi * np.arange(1, k + 1) / k)  # exclude f = 0 (error is 0 there)
    grid = np.linspace(0.0, 1.0, 200001)
    a = np.zeros(degree)
    for _ in range(iters):
        # p(x_i) - 2^x_i = (-1)^i E 2^x_i  ->  sum_j a_j x_i^j - (-1)^i E 2^x_i = 2^x_i - 1
        A = np.zeros((k, k))
        for i, xi in enumerate(x):
            for j in range(degree):
                A[i, j] = xi ** (j + 1)
            A[i, degree] = -((-1) ** i) * 2.0 ** xi
        rhs = 2.0 ** x - 1.0
        sol = np.linalg.solve(A, rhs)
        a = sol[:degree]
        err = (1.0 + sum(a[j] * grid ** (j + 1) for j in range(degree))) / 2.0 ** grid - 1.0
        # new alternation set: extrema of the error between sign changes
        idx = np.where(np.diff(np.sign(np.diff(err))) != 0)[0] + 1
        cand = np.concatenate([idx, [len(grid) - 1]])
        ext = cand[np.argsort(-np.abs(err[cand]))][:k]
        x = np.sort(grid[ext])
    return a


def fp32_horner_error(coef32):
    f = np.linspace(0.0, 1.0, 1 << 20, endpoint=False, dtype=np.float64).astype(np.float32)
    a1, a2, a3 = (np.float32(c) for c in coef32)
    p = np.float32(a3) * f + a2
    p = p.astype(np.float32) * f + a1
    p = p.astype(np.float32) * f + np.float32(1.0)
    p = p.astype(np.float32)
    rel = p.astype(np.float64) / np.exp2(f.astype(np.float64)) - 1.0
    return np.abs(rel).max(), np.abs(rel).mean()


if __name__ == "__main__":
    a = remez(3)
    c32 = [np.float32(v) for v in a]
    mx, mean = fp32_horner_error(c32)
    for i, c in enumerate(c32, 1):
        print(f"a{i} = {float(c)!r}f  (0x{np.float32(c).view(np.uint32):08x})")
    print(f"max rel err {mx:.3e}, mean {mean:.3e}")
