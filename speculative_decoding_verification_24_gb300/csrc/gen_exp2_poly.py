"""Coefficients of the FMA-pipe 2^r polynomial in sv_device.cuh (ex2_poly2).

A minimax polynomial of degree 6 for 2^r on r in [-1/2, 1/2], minimising the
relative error, found with the Remez exchange algorithm in 50-digit
arithmetic (mpmath), then rounded to float32. Run it to reproduce the hex
constants and the error figures quoted beside them:

    python gen_exp2_poly.py

The error of the float32 Horner evaluation (with the x = n + r reduction of
ex2_poly2) is measured here on 6 million arguments in [-126, 0] against
exact 2^x.
"""
import mpmath as mp
import numpy as np

DEG = 6


def remez(deg, a=-0.5, b=0.5, iters=30, grid_pts=4000):
    """Coefficients c[0..deg] of the minimax relative-error fit of 2^x."""
    f = lambda x: mp.power(2, x)  # noqa: E731
    n = deg + 2
    xs = [(a + b) / 2 + (b - a) / 2 * mp.cos(mp.pi * (n - 1 - i) / (n - 1)) for i in range(n)]
    for _ in range(iters):
        A = mp.matrix(n, n)
        rhs = mp.matrix(n, 1)
        for i, x in enumerate(xs):
            for j in range(deg + 1):
                A[i, j] = x ** j
            A[i, deg + 1] = (-1) ** i * f(x)
            rhs[i] = f(x)
        sol = mp.lu_solve(A, rhs)
        c = [sol[j] for j in range(deg + 1)]
        err = lambda x: (sum(c[j] * x ** j for j in range(deg + 1)) - f(x)) / f(x)  # noqa: E731
        grid = [a + (b - a) * mp.mpf(k) / grid_pts for k in range(grid_pts + 1)]
        vals = [err(x) for x in grid]
        ext = [grid[0]] + [grid[k] for k in range(1, grid_pts)
                           if (vals[k] - vals[k - 1]) * (vals[k + 1] - vals[k]) <= 0] + [grid[-1]]
        if len(ext) != n:
            ext = sorted(sorted(ext, key=lambda x: -abs(err(x)))[:n])
        xs = ext
    return c, abs(sol[deg + 1])


def measured_error(c32):
    f32 = lambda v: np.asarray(v, dtype=np.float64).astype(np.float32).astype(np.float64)  # noqa: E731
    rng = np.random.default_rng(0)
    x = f32(np.concatenate([rng.uniform(-126, 0, 4_000_000), rng.uniform(-1, 0, 2_000_000)]))
    M = 12582912.0  # 1.5 * 2^23: x + M rounds x to the nearest integer
    t = f32(x + M)
    n = f32(t - M)
    r = f32(x - n)
    p = np.full_like(r, c32[-1])
    for cj in c32[-2::-1]:
        p = f32(p * r + cj)  # one float32 rounding per step, as fma does
    return float(np.max(np.abs(p * np.exp2(n) - np.exp2(x)) / np.exp2(x)))


if __name__ == "__main__":
    mp.mp.dps = 50
    c, e = remez(DEG)
    c32 = [float(np.float32(float(x))) for x in c]
    print(f"minimax relative error of the exact coefficients: {mp.nstr(e, 5)}")
    print("float32 coefficients c0..c6:", [x.hex() for x in c32])
    print(f"float32 evaluation, max relative error over [-126, 0]: {measured_error(c32):.3e}")
