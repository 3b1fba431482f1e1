"""Fits the polynomial used by the software exp2 in prefill_tc.cu.

exp2(x) is split as 2^n * 2^f with n = round(x) and f = x - n in [-1/2, 1/2]
(Cody-Waite style range reduction; the split is exact in fp32 for the |x| < 2^22 used).
2^f is approximated by a degree-3 polynomial whose coefficients minimise the maximum
RELATIVE error on [-1/2, 1/2], found here with the Remez exchange algorithm in float64.
Run it to reprint the coefficients and the error bound:

    python relative_bias_hybrid_gb300/csrc/fit_exp2_poly.py
"""
import numpy as np


def remez_relative(deg=3, lo=-0.5, hi=0.5, iters=30):
    f = lambda x: np.exp2(x)
    n = deg + 2
    x = 0.5 * (lo + hi) + 0.5 * (hi - lo) * np.cos(np.pi * np.arange(n)[::-1] / (n - 1))
    grid = np.linspace(lo, hi, 200001)
    for _ in range(iters):
        # p(x_i) - f(x_i) = (-1)^i E f(x_i)  (equioscillating relative error)
        A = np.zeros((n, n))
        for i in range(n):
            A[i, :deg + 1] = x[i] ** np.arange(deg + 1)
            A[i, deg + 1] = -((-1) ** i) * f(x[i])
        sol = np.linalg.solve(A, f(x))
        c = sol[:deg + 1]
        err = np.polyval(c[::-1], grid) / f(grid) - 1.0
        # new reference: one extremum per sign-alternating segment
        sign = np.sign(err)
        idx = np.concatenate([[0], np.where(np.diff(sign) != 0)[0] + 1, [len(grid)]])
        ext = [seg_lo + np.argmax(np.abs(err[seg_lo:seg_hi])) for seg_lo, seg_hi in zip(idx[:-1], idx[1:])]
        if len(ext) == n:
            x = grid[np.array(ext)]
    return c, np.abs(err).max()


if __name__ == "__main__":
    c, e = remez_relative()
    c32 = c.astype(np.float32)
    grid = np.linspace(-0.5, 0.5, 1000001)
    p32 = np.polyval(c32.astype(np.float64)[::-1], grid)
    print("coefficients c0..c3 (fp32):", ", ".join(f"{v!r}" for v in c32.tolist()))
    print(f"max relative error: {e:.3e} (float64 coefficients), "
          f"{np.abs(p32 / np.exp2(grid) - 1).max():.3e} (fp32 coefficients)")
