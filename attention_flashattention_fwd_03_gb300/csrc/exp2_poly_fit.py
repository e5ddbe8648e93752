"""Regenerates the coefficients of the degree-3 polynomial that exp2_fma2
(ptx.cuh) uses for 2^f on [-1/2, 1/2].

Method: a minimax fit in relative error by Lawson's iteratively reweighted least
squares (C. L. Lawson, "Contributions to the theory of linear least maximum
approximation", 1961): repeat a weighted least-squares fit, multiplying each
point's weight by its current error, until the error equioscillates.  The
printed error is that of the fp32-rounded coefficients evaluated with fp32
Horner steps.  Run: python exp2_poly_fit.py
"""

import numpy as np


def fit(deg: int = 3, iters: int = 400):
    f = np.linspace(-0.5, 0.5, 20001)
    y = np.exp2(f)
    V = np.vander(f, deg + 1, increasing=True)
    w = np.ones_like(f)
    for _ in range(iters):
        W = np.sqrt(w) / y
        c, *_ = np.linalg.lstsq(V * W[:, None], y * W, rcond=None)
        err = np.abs(V @ c - y) / y
        w = w * err
        w /= w.sum()
    c32 = c.astype(np.float32)
    fx = f.astype(np.float32)
    p = np.float32(c32[-1])
    for k in range(deg - 1, -1, -1):
        p = (p * fx + c32[k]).astype(np.float32)
    return c32, float(np.max(np.abs(p.astype(np.float64) - y) / y))


if __name__ == "__main__":
    coeffs, rel = fit()
    print("c0..c3 =", [float(x) for x in coeffs], "max relative error", rel)
