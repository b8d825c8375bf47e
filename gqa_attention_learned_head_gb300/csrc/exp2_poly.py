"""Derives the polynomial that the prefill softmax uses for part of its exp2 evaluations.

2^x is split as 2^round(x) * 2^f with f = x - round(x) in [-1/2, 1/2]; 2^f is approximated by a
cubic p(f) = c0 + c1 f + c2 f^2 + c3 f^3 chosen to minimise the maximum RELATIVE error on
[-1/2, 1/2] (a Remez-style exchange on the relative error, started from a Chebyshev-node least
squares fit).  The result is rounded to float32 and printed as C constants; the relative error
(~1e-4) is far below bf16's 2^-9 rounding of the probabilities that feed P.V.

    python exp2_poly.py
"""
import numpy as np


def fit(deg=3, iters=30):
    a, b = -0.5, 0.5
    n = deg + 2
    # start: least squares on Chebyshev nodes, relative weights
    xs = 0.5 * (a + b) + 0.5 * (b - a) * np.cos(np.pi * (np.arange(200) + 0.5) / 200)
    A = np.vander(xs, deg + 1, increasing=True) / (2.0 ** xs)[:, None]
    c = np.linalg.lstsq(A, np.ones_like(xs), rcond=None)[0]
    ref = np.linspace(a, b, n)
    grid = np.linspace(a, b, 20001)
    for _ in range(iters):
        # solve p(x_i) / 2^x_i - 1 = (-1)^i E on the reference set
        M = np.zeros((n, n))
        M[:, :deg + 1] = np.vander(ref, deg + 1, increasing=True) / (2.0 ** ref)[:, None]
        M[:, deg + 1] = (-1.0) ** np.arange(n)
        sol = np.linalg.solve(M, np.ones(n))
        c = sol[:deg + 1]
        err = np.polyval(c[::-1], grid) / 2.0 ** grid - 1.0
        # new reference: extrema of the error between sign changes
        idx = [0]
        for i in range(1, len(grid) - 1):
            if (err[i] - err[i - 1]) * (err[i + 1] - err[i]) <= 0:
                idx.append(i)
        idx.append(len(grid) - 1)
        cand = sorted(idx, key=lambda i: -abs(err[i]))
        chosen = sorted(cand[:n])
        if len(chosen) == n:
            ref = grid[chosen]
    return c.astype(np.float32)


def max_rel_error(c):
    g = np.linspace(-0.5, 0.5, 200001)
    p = ((np.float64(c[3]) * g + c[2]) * g + c[1]) * g + c[0]
    return float(np.max(np.abs(p / 2.0 ** g - 1.0)))


if __name__ == "__main__":
    c = fit()
    for i, v in enumerate(c):
        print(f"constexpr float kExp2C{i} = {float(v)!r}f;")
    print(f"// max relative error on [-1/2, 1/2]: {max_rel_error(c):.3e}")
