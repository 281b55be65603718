"""Fit the polynomial used by exp2_poly3() in ptx.cuh.

2^x is split as 2^n * 2^f with n = round(x) and f = x - n in [-0.5, 0.5]
(Cody and Waite's range reduction); 2^f is approximated by a cubic whose
coefficients minimise the maximum RELATIVE error on [-0.5, 0.5] (Lawson's
iteratively reweighted least squares converging to the minimax fit).  The
kernel rounds the result to bf16 (8-bit significand) or tf32 (11-bit), so a
relative error near 1e-4 is far below what those formats keep.

Run:  python fit_exp2_poly.py   (prints the coefficients and the error bound)
"""
import numpy as np


def fit(degree: int = 3, lo: float = -0.5, hi: float = 0.5, iters: int = 400):
    x = np.linspace(lo, hi, 40001)
    y = np.exp2(x)
    A = np.vander(x, degree + 1, increasing=True)
    w = np.full_like(x, 1.0 / x.size)
    for _ in range(iters):
        W = np.sqrt(w) / y
        c, *_ = np.linalg.lstsq(A * W[:, None], y * W, rcond=None)
        e = np.abs(A @ c - y) / y
        w = w * e
        w /= w.sum()
    c = c.astype(np.float32).astype(np.float64)  # what the kernel will hold
    err = float(np.max(np.abs(A @ c - y) / y))
    return c, err


if __name__ == "__main__":
    c, err = fit()
    for i, ci in enumerate(c):
        print(f"c{i} = {np.float32(ci)!r}  ({float(np.float32(ci)).hex()})")
    print(f"max relative error on [-0.5, 0.5]: {err:.3e} (2^{np.log2(err):.2f})")
