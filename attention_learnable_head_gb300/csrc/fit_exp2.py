"""Fit the polynomial used for the FMA-pipe exp2 in the forward softmax.

2^x is split Cody-Waite style into 2^n * 2^f with n = round(x) and
f = x - n in [-1/2, 1/2]; 2^f is approximated by a polynomial p(f) whose
coefficients minimise the maximum relative error on that interval.  The fit
is a least-squares fit on Chebyshev nodes refined by Lawson's iteratively
reweighted scheme, which converges to the minimax (equioscillating) solution.
Coefficients are then rounded to fp32 and the error re-measured in fp32
Horner evaluation.

    python fit_exp2.py [degree]
"""
import sys

import numpy as np


def fit(degree: int, nodes: int = 4000, iters: int = 400):
    f = np.cos(np.pi * (np.arange(nodes) + 0.5) / nodes) * 0.5      # Chebyshev nodes in [-1/2, 1/2]
    target = np.exp2(f)
    V = np.vander(f, degree + 1, increasing=True) / target[:, None]   # relative error
    w = np.ones(nodes) / nodes
    for _ in range(iters):
        sw = np.sqrt(w)
        c, *_ = np.linalg.lstsq(V * sw[:, None], sw, rcond=None)
        err = np.abs(V @ c - 1.0)
        w = w * err
        w /= w.sum()
    return c


def max_rel_error_fp32(c):
    f = np.linspace(-0.5, 0.5, 200001).astype(np.float32)
    cf = c.astype(np.float32)
    p = np.full_like(f, cf[-1])
    for a in cf[-2::-1]:
        p = (p * f + a).astype(np.float32)
    return float(np.max(np.abs(p.astype(np.float64) / np.exp2(f.astype(np.float64)) - 1.0)))


if __name__ == "__main__":
    deg = int(sys.argv[1]) if len(sys.argv) > 1 else 3
    c = fit(deg)
    print("degree", deg, "coefficients (c0..cn):")
    for a in c:
        print(f"  {np.float32(a)!r}  ({a:.17g})")
    print("max relative error (fp32 Horner):", max_rel_error_fp32(c))
