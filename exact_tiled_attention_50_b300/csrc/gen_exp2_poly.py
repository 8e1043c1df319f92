"""Coefficients of the cubic that approximates 2^f on [-1/2, 1/2] in the softmax kernel.

The kernel evaluates some of its exponentials on the FMA pipe as 2^x = 2^n * p(f), with
n = round(x), f = x - n, p(f) = c0 + c1 f + c2 f^2 + c3 f^3. The cubic minimises the maximum
relative error |p(f) / 2^f - 1| over the interval (equi-oscillation found by a Remez exchange on a
dense grid). Run this file to print the coefficients as fp32 literals and the error bound.
"""
import numpy as np


def remez_relative(deg=3, lo=-0.5, hi=0.5, iters=30):
    grid = np.linspace(lo, hi, 20001)
    target = np.exp2(grid)
    # start from Chebyshev extrema
    k = np.arange(deg + 2)
    pts = 0.5 * (lo + hi) + 0.5 * (hi - lo) * np.cos(np.pi * k[::-1] / (deg + 1))
    for _ in range(iters):
        # solve p(x_i) - 2^x_i = (-1)^i E 2^x_i  (relative equi-oscillation)
        A = np.zeros((deg + 2, deg + 2))
        for i, x in enumerate(pts):
            A[i, :deg + 1] = x ** np.arange(deg + 1)
            A[i, deg + 1] = -((-1) ** i) * np.exp2(x)
        sol = np.linalg.solve(A, np.exp2(pts))
        c = sol[:deg + 1]
        err = np.polyval(c[::-1], grid) / target - 1.0
        # new reference: one extremum per sign run
        sign = np.sign(err)
        runs = np.split(np.arange(len(grid)), np.where(np.diff(sign) != 0)[0] + 1)
        ext = [r[np.argmax(np.abs(err[r]))] for r in runs]
        if len(ext) != deg + 2:
            break
        pts = grid[ext]
    return c, np.max(np.abs(err))


if __name__ == "__main__":
    c, e = remez_relative()
    c32 = np.float32(c)
    f = np.linspace(-0.5, 0.5, 200001, dtype=np.float64)
    p = ((c32[3].astype(np.float64) * f + c32[2]) * f + c32[1]) * f + c32[0]
    print("coefficients c0..c3:", ", ".join(f"{float(v)!r}f" for v in c32))
    print(f"max relative error of the fp32 cubic on [-1/2, 1/2]: {np.max(np.abs(p / np.exp2(f) - 1)):.3e}")
