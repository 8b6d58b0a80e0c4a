"""Derives the coefficients of the polynomial exp2 used on the FMA pipes.

Method (Cody-Waite range reduction plus a minimax polynomial): write
x = n + f with n = round(x) and f in [-1/2, 1/2]; then 2^x = 2^n * 2^f, where
2^n is applied by adding n to the float's exponent field and 2^f is a
polynomial p(f).  The coefficients below minimise max |p(f) / 2^f - 1| over
[-1/2, 1/2] (Lawson's iteratively reweighted least squares, which converges to
the minimax fit), then are rounded to float32 and re-checked in float32
arithmetic with the Horner order the kernels use.

Run:  python exp2_poly_fit.py [degree]
Prints the coefficients (c0 first) and the worst relative error.
"""
import sys

import numpy as np


def fit(degree: int, iters: int = 200, n_grid: int = 20001):
    f = np.linspace(-0.5, 0.5, n_grid)
    target = np.exp2(f)
    A = np.vander(f, degree + 1, increasing=True) / target[:, None]  # relative error basis
    b = np.ones_like(f)
    w = np.full(n_grid, 1.0 / n_grid)
    c = None
    for _ in range(iters):
        sw = np.sqrt(w)
        c, *_ = np.linalg.lstsq(A * sw[:, None], b * sw, rcond=None)
        err = np.abs(A @ c - b)
        w = w * err
        w /= w.sum()
    return c


def check_f32(c, n=2_000_001):
    """Evaluates the kernels' float32 sequence (clamp at -126, round by the
    1.5 * 2^23 shift, Horner, exponent add) on [-130, 0]; returns the worst
    relative error on [-125, 0] (below that the result can land in the
    denormal encoding) and asserts that below -125 the result is a finite
    value in [0, 2^-124]."""
    c32 = np.asarray(c, np.float32)
    x = np.maximum(np.linspace(-130.0, 0.0, n).astype(np.float32), np.float32(-126.0))
    xin = np.linspace(-130.0, 0.0, n)
    magic = np.float32(12582912.0)  # 1.5 * 2^23: adding it rounds to an integer
    t = (x + magic).astype(np.float32)
    nf = (t - magic).astype(np.float32)
    fr = (x - nf).astype(np.float32)
    p = c32[-1]
    for k in range(len(c32) - 2, -1, -1):
        p = (p * fr + c32[k]).astype(np.float32)
    bits = (p.view(np.uint32) + (t.view(np.uint32) << np.uint32(23))).astype(np.uint32)
    y = bits.view(np.float32).astype(np.float64)
    low = xin < -125.0
    assert np.all(np.isfinite(y)) and np.all(y[low] >= 0.0) and np.all(y[low] <= 2.0 ** -124)
    ref = np.exp2(xin)
    ok = xin >= -125.0
    return c32, float(np.max(np.abs(y[ok] / ref[ok] - 1.0)))


if __name__ == "__main__":
    deg = int(sys.argv[1]) if len(sys.argv) > 1 else 3
    c = fit(deg)
    c32, err = check_f32(c)
    print("coefficients:", ", ".join(f"{v:.9e}f" for v in c32))
    print(f"max relative error (float32 evaluation, x in [-125, 0]): {err:.3e}; below -125: finite, in [0, 2^-124]")
