"""Coefficients of the FMA-pipe 2^f used by the fused forward's softmax.

2^x is split Cody-Waite style as x = n + f with n = round(x) and f in
[-1/2, 1/2]; 2^n goes into the exponent field and 2^f is a degree-3
polynomial.  The coefficients below minimise the maximum RELATIVE error
|p(f) / 2^f - 1| on [-1/2, 1/2] (Remez exchange on the equioscillation
points), with p(0) free.  Run this file to reproduce them:

    python optimal_tiling_gb300/csrc/gen_exp2_poly.py
"""
import numpy as np


def remez_rel(deg=3, lo=-0.5, hi=0.5, iters=30):
    f = lambda x: np.exp2(x)
    # start from Chebyshev extrema
    k = np.arange(deg + 2)
    xs = (lo + hi) / 2 + (hi - lo) / 2 * np.cos(np.pi * k[::-1] / (deg + 1))
    grid = np.linspace(lo, hi, 200001)
    for _ in range(iters):
        # solve p(x_i) - f(x_i) = (-1)^i E f(x_i)  (relative weight)
        A = np.zeros((deg + 2, deg + 2))
        for i, x in enumerate(xs):
            A[i, :deg + 1] = [x ** j for j in range(deg + 1)]
            A[i, deg + 1] = -((-1) ** i) * f(x)
        sol = np.linalg.solve(A, f(xs))
        c = sol[:deg + 1]
        err = (np.polyval(c[::-1], grid) - f(grid)) / f(grid)
        # new extrema: one per sign-alternating segment
        idx = [0]
        sgn = np.sign(err)
        seg_starts = [0] + list(np.where(np.diff(sgn) != 0)[0] + 1) + [len(grid)]
        ext = []
        for a, b in zip(seg_starts[:-1], seg_starts[1:]):
            j = a + int(np.argmax(np.abs(err[a:b])))
            ext.append(j)
        if len(ext) != deg + 2:
            # keep the deg+2 largest alternating extrema
            ext = sorted(ext, key=lambda j: -abs(err[j]))[:deg + 2]
            ext.sort()
        xs = grid[ext]
    return c, float(np.max(np.abs(err)))


if __name__ == "__main__":
    c, e = remez_rel()
    c32 = np.float32(c)
    print("coefficients (c0..c3):", ", ".join(f"{float(x):.9e}f" for x in c32))
    print("max relative error:", e)
