"""Coefficients of the polynomial exp2 used by the prefill softmax.

2^x is split as 2^n * 2^f with n = round(x) and f = x - n in [-1/2, 1/2]
(Cody and Waite's range reduction).  2^f is approximated by a cubic whose
coefficients minimise the maximum relative error on [-1/2, 1/2]; the minimax
fit is found with Lawson's algorithm (iteratively reweighted least squares:
the weights of the points with the largest error grow until the error
equioscillates).  The result is good to about 1e-4 relative, far below the
2^-9 rounding that the bf16 P matrix applies afterwards.

Run this file to print the coefficients that exp2_poly.cuh holds.
"""
import numpy as np

DEGREE = 3


def fit(degree=DEGREE, points=4001, iters=200):
    f = np.linspace(-0.5, 0.5, points)
    target = np.exp2(f)
    A = np.vander(f, degree + 1, increasing=True) / target[:, None]   # relative error rows
    b = np.ones_like(f)
    w = np.full(points, 1.0 / points)
    for _ in range(iters):
        sw = np.sqrt(w)
        c, *_ = np.linalg.lstsq(A * sw[:, None], b * sw, rcond=None)
        err = np.abs(A @ c - b)
        w = w * err
        w /= w.sum()
    return c


def max_rel_error(coeffs, points=200001):
    """Max relative error of the float32 evaluation (Horner) against exp2."""
    f = np.linspace(-0.5, 0.5, points).astype(np.float32)
    c = [np.float32(x) for x in coeffs]
    acc = np.full_like(f, c[-1])
    for k in range(len(c) - 2, -1, -1):
        acc = acc * f + c[k]
    return float(np.max(np.abs(acc.astype(np.float64) / np.exp2(f.astype(np.float64)) - 1.0)))


if __name__ == "__main__":
    coeffs = fit()
    for k, c in enumerate(coeffs):
        print("c%d = %.9ef" % (k, np.float32(c)))
    print("max relative error (fp32 Horner): %.3e" % max_rel_error(coeffs))
