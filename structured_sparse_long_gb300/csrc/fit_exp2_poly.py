"""Fits the degree-3 polynomial p(f) ~ 2^f on [-1/2, 1/2] used by exp2_poly() in pi_fwd_tc.cu.

2^x = 2^n * 2^f with n = round(x) and f = x - n in [-1/2, 1/2] (Cody-Waite style range
reduction); 2^f comes from this polynomial and 2^n is added into the exponent field.
The fit is an iteratively re-weighted least-squares fit of the relative error on
Chebyshev nodes, which approaches the equi-oscillating (minimax) solution.

Run:  python structured_sparse_long_gb300/csrc/fit_exp2_poly.py
Prints the fp32 coefficients c0..c3 (low to high order) and the maximum relative error.
"""
import numpy as np


def fit(deg=3, iters=60):
    f = np.cos(np.linspace(0, np.pi, 4001)) * 0.5
    y = 2.0 ** f
    A = np.vander(f, deg + 1, increasing=True)
    w = np.ones_like(f)
    for _ in range(iters):
        c, *_ = np.linalg.lstsq(A * (w / y)[:, None], w, rcond=None)
        err = (A @ c - y) / y
        w = w * (1 + 5 * np.abs(err) / np.abs(err).max())
    c32 = c.astype(np.float32)
    xs = np.linspace(-0.5, 0.5, 200001)
    rel = np.abs(np.polyval(c32.astype(np.float64)[::-1], xs) / 2.0 ** xs - 1).max()
    return c32, rel


if __name__ == "__main__":
    c, rel = fit()
    print("coefficients:", ", ".join(f"{float(x)!r}f" for x in c))
    print("max relative error on [-0.5, 0.5]:", rel)
