"""Fit the polynomial the prefill kernel uses for part of its exponentials.

2^x = 2^n * 2^f with n = round(x) and f = x - n in [-1/2, 1/2] (range reduction: the
integer part goes into the exponent field, the fractional part into a polynomial).  This
script fits p(f) ~ 2^f of the given degree minimising the maximum RELATIVE error on
[-1/2, 1/2] by the Remez exchange algorithm (equioscillation at degree + 2 points), in
float64, and prints the coefficients as float32 values together with the relative error
of the float32 Horner evaluation.  The kernel's constants are this script's output;
tests/test_exp2_poly.py checks them against the error bound printed here.

    python head_aware_paged_rope_b300/csrc/fit_exp2.py [degree]
"""
import sys

import numpy as np


def remez(deg, lo=-0.5, hi=0.5, iters=40):
    n = deg + 2
    # Chebyshev extrema as the starting reference
    x = np.sort((lo + hi) / 2 + (hi - lo) / 2 * np.cos(np.pi * np.arange(n) / (n - 1)))
    grid = np.linspace(lo, hi, 200001)
    for _ in range(iters):
        # solve  p(x_i) - 2^x_i = (-1)^i E 2^x_i  for the coefficients and E (relative error)
        A = np.zeros((n, n))
        for i, xi in enumerate(x):
            A[i, :deg + 1] = xi ** np.arange(deg + 1)
            A[i, deg + 1] = (-1) ** i * 2.0 ** xi
        sol = np.linalg.solve(A, 2.0 ** x)
        c = sol[:deg + 1]
        err = (np.polyval(c[::-1], grid) - 2.0 ** grid) / 2.0 ** grid
        # new reference: the extrema of the error between its sign changes
        s = np.sign(err)
        idx = np.concatenate([[0], np.nonzero(np.diff(s))[0] + 1, [len(grid)]])
        ext = [grid[a + np.argmax(np.abs(err[a:b]))] for a, b in zip(idx[:-1], idx[1:]) if b > a]
        if len(ext) >= n:
            # keep the n largest alternating extrema
            ext = np.array(ext)
            while len(ext) > n:
                e = np.abs((np.polyval(c[::-1], ext) - 2.0 ** ext) / 2.0 ** ext)
                drop = 0 if e[0] < e[-1] else len(ext) - 1
                ext = np.delete(ext, drop)
            x = np.sort(ext)
    return c, np.abs(err).max()


def horner_f32(c32, f):
    p = np.float32(c32[-1]) * np.ones_like(f, dtype=np.float32)
    for ck in c32[-2::-1]:
        p = (p * f + np.float32(ck)).astype(np.float32)   # the kernel uses fused multiply-adds
    return p


if __name__ == "__main__":
    deg = int(sys.argv[1]) if len(sys.argv) > 1 else 3
    c, e64 = remez(deg)
    c32 = c.astype(np.float32)
    f = np.linspace(-0.5, 0.5, 1000001).astype(np.float32)
    rel = np.abs(horner_f32(c32, f).astype(np.float64) / 2.0 ** f.astype(np.float64) - 1).max()
    print(f"degree {deg}: minimax relative error {e64:.3e} (float64), {rel:.3e} with float32 coefficients")
    for k, v in enumerate(c32):
        print(f"  c{k} = {float(v)!r}f  ({v.view(np.uint32):#010x})")
