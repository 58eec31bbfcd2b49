"""Coefficients of the FMA-pipe 2^f polynomial used by the statistics pass.

The statistics pass evaluates part of its exponentials without the MUFU unit:
t = j + f with j = rint(t) and |f| <= 1/2 (Cody and Waite's argument
reduction), 2^f from a degree-6 polynomial, 2^j added to the exponent field.
This script fits the polynomial by the Remez exchange algorithm on the
relative error over [-1/2, 1/2], rounds the coefficients to fp32, and reports
the worst relative error of the fp32 Horner evaluation on a dense grid.  Its
output is pasted into sv_common.cuh (exp2_poly2).

    python gen_exp2_poly.py
"""
import numpy as np


def remez_relative(deg, a=-0.5, b=0.5, iters=40, grid=400001):
    n = deg + 2
    x = 0.5 * (a + b) + 0.5 * (b - a) * np.cos(np.pi * np.arange(n)[::-1] / (n - 1))
    t = np.linspace(a, b, grid)
    coef = None
    for _ in range(iters):
        A = np.zeros((n, n))
        for i, xi in enumerate(x):
            A[i, :deg + 1] = xi ** np.arange(deg + 1)
            A[i, deg + 1] = -((-1) ** i) * np.exp2(xi)
        sol = np.linalg.solve(A, np.exp2(x))
        coef = sol[:deg + 1]
        err = (np.polyval(coef[::-1], t) - np.exp2(t)) / np.exp2(t)
        # alternating extrema of the error
        idx = [0]
        for i in range(1, len(t)):
            if np.sign(err[i]) != np.sign(err[idx[-1]]):
                idx.append(i)
            elif abs(err[i]) > abs(err[idx[-1]]):
                idx[-1] = i
        while len(idx) > n:
            if abs(err[idx[0]]) < abs(err[idx[-1]]):
                idx.pop(0)
            else:
                idx.pop()
        if len(idx) == n:
            x = t[idx]
    return coef


def horner_f32(c32, t):
    p = np.full_like(t, c32[-1])
    for k in range(len(c32) - 2, -1, -1):
        p = (p * t + c32[k]).astype(np.float32)
    return p


if __name__ == "__main__":
    coef = remez_relative(6)
    c32 = coef.astype(np.float32)
    t = np.linspace(-0.5, 0.5, 4000001).astype(np.float32)
    p = horner_f32(c32, t).astype(np.float64)
    ref = np.exp2(t.astype(np.float64))
    print("max relative error of the fp32 evaluation: %.3g" % (np.abs(p - ref) / ref).max())
    for k, c in enumerate(c32):
        print(f"  c{k} = {float(c).hex()}f  // {float(c)!r}")
