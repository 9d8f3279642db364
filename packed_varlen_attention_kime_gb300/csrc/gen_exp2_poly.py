"""Derives the coefficients of exp2_poly (kime_common.cuh): the degree-3
polynomial minimising the maximum relative error of 2^f on [-0.5, 0.5], by the
Remez exchange algorithm.  Run it to print the coefficients and the error.

2^x is evaluated as 2^n * 2^f with n = round(x), f = x - n in [-0.5, 0.5]
(Cody-Waite style argument reduction; the 2^n factor is an exponent-field
add), so only 2^f needs a polynomial.
"""
import numpy as np


def remez(deg, a=-0.5, b=0.5, iters=60, grid=200001):
    n = deg + 2
    x = 0.5 * (a + b) + 0.5 * (b - a) * np.cos(np.pi * np.arange(n)[::-1] / (n - 1))
    g = np.linspace(a, b, grid)
    for _ in range(iters):
        # solve p(x_i) + (-1)^i E 2^x_i = 2^x_i  (equioscillating relative error)
        A = np.zeros((n, n))
        for i, xi in enumerate(x):
            A[i, : deg + 1] = xi ** np.arange(deg + 1)
            A[i, deg + 1] = (-1) ** i * 2.0 ** xi
        c = np.linalg.solve(A, 2.0 ** x)[: deg + 1]
        err = (np.polyval(c[::-1], g) - 2.0 ** g) / 2.0 ** g
        # one extremum per sign run
        idx = [0]
        for k in range(1, len(g)):
            if np.sign(err[k]) != np.sign(err[idx[-1]]):
                idx.append(k)
            elif abs(err[k]) > abs(err[idx[-1]]):
                idx[-1] = k
        if len(idx) >= n:
            x = g[idx[:n]]
    return c, float(np.max(np.abs(err)))


if __name__ == "__main__":
    c, e = remez(3)
    print("coefficients (c0..c3):", [float(np.float32(v)) for v in c])
    print("max relative error on [-0.5, 0.5]:", e)
