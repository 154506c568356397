"""Fits the polynomial used by the kernels' FMA-pipe exp2.

2^f on [0, 1) is approximated by p(f) = 1 + c1 f + c2 f^2 + c3 f^3 (the constant
term is pinned to 1 so that p(0) = 1 exactly, as the FlashAttention-4 summary,
section 3.1.3, describes). The coefficients minimise the maximum relative
error (minimax) and are found with a Remez exchange on the relative error, in
float64, then rounded to float32. Run as a script to print them; the values are
the constants of ``exp2_poly3_x2`` in ``attn_common.cuh``.
"""

import numpy as np


def _rel_err(c, f):
    p = 1.0 + f * (c[0] + f * (c[1] + f * c[2]))
    return p / np.exp2(f) - 1.0


def remez(deg=3, iters=30):
    n = deg  # unknown coefficients c1..c_deg, plus the level E
    # initial reference: n + 1 Chebyshev-like points in (0, 1]; f = 0 is excluded
    # because p(0) = 1 makes the error vanish there
    k = np.arange(1, n + 2)
    x = 0.5 - 0.5 * np.cos(np.pi * k / (n + 1))
    grid = np.linspace(0.0, 1.0, 200001)[1:]
    c = np.zeros(n)
    for _ in range(iters):
        # solve p(x_i)/2^x_i - 1 = (-1)^i E  for c and E
        a = np.zeros((n + 1, n + 1))
        rhs = np.zeros(n + 1)
        for i, xi in enumerate(x):
            w = 1.0 / np.exp2(xi)
            for j in range(n):
                a[i, j] = w * xi ** (j + 1)
            a[i, n] = -((-1.0) ** i)
            rhs[i] = 1.0 - w
        sol = np.linalg.solve(a, rhs)
        c = sol[:n]
        e = _rel_err(c, grid)
        # new reference: alternating extrema of the error
        sign = np.sign(e)
        idx = [0]
        for i in range(1, len(grid)):
            if sign[i] != sign[idx[-1]]:
                idx.append(i)
            elif abs(e[i]) > abs(e[idx[-1]]):
                idx[-1] = i
        if len(idx) < n + 1:
            break
        # keep n + 1 consecutive extrema with the largest minimum
        best = None
        for s in range(len(idx) - n):
            cand = idx[s:s + n + 1]
            m = min(abs(e[i]) for i in cand)
            if best is None or m > best[0]:
                best = (m, cand)
        x = grid[best[1]]
    return c, float(np.max(np.abs(_rel_err(c, grid))))


if __name__ == "__main__":
    c, err = remez(3)
    c32 = c.astype(np.float32)
    grid = np.linspace(0.0, 1.0, 1000001, dtype=np.float64)
    err32 = float(np.max(np.abs(_rel_err(c32.astype(np.float64), grid))))
    print("coefficients c1..c3 (float32):", [float(v) for v in c32])
    print("hex:", [hex(np.float32(v).view(np.uint32)) for v in c32])
    print(f"max relative error: float64 coefficients {err:.3e}, float32 coefficients {err32:.3e}")
