"""Fit the polynomial the prefill kernel uses for part of its exp2 evaluations.

Method: Cody-Waite style range reduction in base 2 (2^x = 2^j * 2^f with
j = round(x), f = x - j in [-1/2, 1/2]; the reduction is exact because the base
is 2) followed by a polynomial p(f) ~= 2^f of degree n whose coefficients
minimise the maximum relative error on [-1/2, 1/2] (minimax, found with the
Remez exchange algorithm in 50-digit arithmetic), then rounded to float32.

The script prints the float32 coefficients (c0 .. cn, increasing powers) and
the maximum relative error of the float32 Horner evaluation with fused
multiply-adds, measured on a dense grid.  Run: python fit_exp2.py [degree]
"""
import sys

import mpmath as mp
import numpy as np


def remez(n, a=-0.5, b=0.5, iters=30):
    """Minimax polynomial of degree n for 2^x on [a, b], relative error."""
    mp.mp.dps = 50
    f = lambda x: mp.power(2, x)
    # start from Chebyshev extrema
    m = n + 2
    xs = [mp.mpf(a + b) / 2 + mp.mpf(b - a) / 2 * mp.cos(mp.pi * i / (m - 1)) for i in range(m)][::-1]
    coef = None
    for _ in range(iters):
        # solve sum c_k x_i^k + (-1)^i E f(x_i) = f(x_i)
        A = mp.matrix(m, m)
        rhs = mp.matrix(m, 1)
        for i, x in enumerate(xs):
            for k in range(n + 1):
                A[i, k] = x ** k
            A[i, n + 1] = (-1) ** i * f(x)
            rhs[i] = f(x)
        sol = mp.lu_solve(A, rhs)
        coef = [sol[k] for k in range(n + 1)]
        err = lambda x: (mp.polyval(coef[::-1], x) - f(x)) / f(x)
        # new reference: extrema of the error on a fine grid
        grid = [mp.mpf(a) + (mp.mpf(b) - a) * i / 4000 for i in range(4001)]
        vals = [err(x) for x in grid]
        ext = [grid[0]]
        for i in range(1, len(grid) - 1):
            if (vals[i] - vals[i - 1]) * (vals[i + 1] - vals[i]) <= 0:
                ext.append(grid[i])
        ext.append(grid[-1])
        # keep m alternating extrema with the largest magnitudes
        ev = [err(x) for x in ext]
        pick = []
        for x, e in zip(ext, ev):
            if pick and mp.sign(e) == mp.sign(pick[-1][1]):
                if abs(e) > abs(pick[-1][1]):
                    pick[-1] = (x, e)
            else:
                pick.append((x, e))
        while len(pick) > m:
            if abs(pick[0][1]) < abs(pick[-1][1]):
                pick.pop(0)
            else:
                pick.pop()
        if len(pick) < m:
            break
        xs = [x for x, _ in pick]
    return coef


def eval_f32(c32, x):
    """Float32 Horner evaluation with fused multiply-add (one rounding per step)."""
    x = np.asarray(x, dtype=np.float32)
    p = np.full_like(x, c32[-1])
    for c in c32[-2::-1]:
        p = (p.astype(np.float64) * x.astype(np.float64) + np.float64(c)).astype(np.float32)
    return p


def main():
    n = int(sys.argv[1]) if len(sys.argv) > 1 else 5
    coef = remez(n)
    c32 = np.array([float(c) for c in coef], dtype=np.float32)
    x = np.linspace(-0.5, 0.5, 2000001, dtype=np.float64).astype(np.float32)
    rel = np.abs(eval_f32(c32, x).astype(np.float64) / np.exp2(x.astype(np.float64)) - 1.0)
    print("degree", n)
    for i, c in enumerate(c32):
        print("  c%d = %.9e  (0x%08x)" % (i, c, c.view(np.uint32)))
    print("max relative error of the float32 evaluation on [-1/2, 1/2]: %.3e (%.2f ulp of 1.0)"
          % (rel.max(), rel.max() / 2.0 ** -23))


if __name__ == "__main__":
    main()
