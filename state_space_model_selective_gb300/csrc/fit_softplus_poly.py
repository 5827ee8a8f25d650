"""Derivation of the polynomial in softplus_f (common.cuh).

softplus(x) = max(x, 0) + log1p(t), t = exp(-|x|) in (0, 1].  With
s = t / (2 + t) in (0, 1/3], log1p(t) = 2 atanh(s) = 2 s f(s^2) where
f(w) = atanh(sqrt(w)) / sqrt(w) = 1 + w/3 + w^2/5 + ...  on w in [0, 1/9].
This script fits a degree-4 polynomial to f minimising the maximum relative
error (Lawson-reweighted least squares on Chebyshev nodes) and prints the
coefficients in fp32 and the error of their fp32 Horner evaluation.
"""
import numpy as np


def f(w):
    s = np.sqrt(w)
    out = np.ones_like(w)
    m = w > 0
    out[m] = np.arctanh(s[m]) / s[m]
    return out


def fit(deg=4, wmax=1.0 / 9.0, iters=60):
    x = (np.cos(np.linspace(0, np.pi, 400)) + 1) / 2 * wmax
    wts = np.ones_like(x)
    for _ in range(iters):
        V = np.vander(x, deg + 1, increasing=True)
        c, *_ = np.linalg.lstsq(V * (wts / f(x))[:, None], wts, rcond=None)
        err = (V @ c - f(x)) / f(x)
        wts = wts * np.sqrt(np.abs(err) + 1e-30)
        wts /= wts.max()
    return c.astype(np.float32)


if __name__ == "__main__":
    c = fit()
    xx = np.linspace(0, 1.0 / 9.0, 200001).astype(np.float32)
    p = np.full_like(xx, c[-1])
    for k in range(len(c) - 2, -1, -1):
        p = (p * xx + c[k]).astype(np.float32)
    err = np.max(np.abs((p.astype(np.float64) - f(xx.astype(np.float64))) / f(xx.astype(np.float64))))
    print("coefficients (w^0 .. w^4):", [float(v) for v in c])
    print("max relative error of the fp32 evaluation:", err)
