"""Fit the polynomial of the softmax warps' FMA-pipe exp2.

exp2(x) is split as x = j + f with j = round(x) and f in [-1/2, 1/2] (Cody and
Waite's additive range reduction); 2^j is put into the float's exponent field
and 2^f is approximated by a degree-3 polynomial p(f) whose coefficients
minimise the maximum relative error max |p(f) / 2^f - 1| on [-1/2, 1/2].  The
fit is a plain Remez exchange on the relative-error weight, in 80-bit-free
double precision with mpmath for the reference values.

Run:  python fit_exp2_poly.py      -> prints the coefficients (float32) and the error.
The kernel's EXP2_C0..C3 constants are this script's output.
"""
import mpmath as mp
import numpy as np

mp.mp.dps = 40
DEG = 3
LO, HI = -0.5, 0.5


def target(x):
    return mp.power(2, x)


def remez(deg=DEG, iters=30):
    n = deg + 2
    # Chebyshev extrema as the initial reference set
    xs = [mp.mpf((LO + HI) / 2 + (HI - LO) / 2 * mp.cos(mp.pi * k / (n - 1))) for k in range(n)][::-1]
    coeffs = None
    for _ in range(iters):
        # solve p(x_k) - 2^x_k = (-1)^k E 2^x_k   (relative weight)
        A = mp.matrix(n, n)
        b = mp.matrix(n, 1)
        for k, x in enumerate(xs):
            for p in range(deg + 1):
                A[k, p] = x ** p
            A[k, deg + 1] = -((-1) ** k) * target(x)
            b[k] = target(x)
        sol = mp.lu_solve(A, b)
        coeffs = [sol[p] for p in range(deg + 1)]

        def rel(x):
            return (sum(c * x ** p for p, c in enumerate(coeffs)) - target(x)) / target(x)
        # new reference: extrema of the relative error on a fine grid, one per sign run
        grid = [mp.mpf(LO + (HI - LO) * t / 4000) for t in range(4001)]
        vals = [rel(x) for x in grid]
        runs, cur = [], [0]
        for t in range(1, len(grid)):
            if mp.sign(vals[t]) == mp.sign(vals[cur[0]]):
                cur.append(t)
            else:
                runs.append(cur)
                cur = [t]
        runs.append(cur)
        ext = [max(r, key=lambda t: abs(vals[t])) for r in runs]
        if len(ext) != n:
            break
        xs = [grid[t] for t in ext]
    return coeffs


def max_rel_error_f32(c):
    """Max relative error of the float32 Horner evaluation over a dense grid of [-1/2, 1/2]."""
    f = np.linspace(LO, HI, 200001, dtype=np.float32)
    c32 = [np.float32(float(x)) for x in c]
    p = np.float32(c32[3])
    for k in (2, 1, 0):
        p = (p * f + c32[k]).astype(np.float32)
    ref = np.exp2(f.astype(np.float64))
    return float(np.max(np.abs(p.astype(np.float64) / ref - 1)))


if __name__ == "__main__":
    c = remez()
    for k, x in enumerate(c):
        print(f"EXP2_C{k} = {float(mp.mpf(x)):.9e}f")
    print("max relative error (float32 Horner):", max_rel_error_f32(c))
