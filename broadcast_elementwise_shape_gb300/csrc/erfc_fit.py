#!/usr/bin/env python
"""Coefficients of the shorter erfc used for GeLU results stored as bfloat16.

The form is that of W. H. Press et al., "Numerical Recipes", section 6.2:
erfc(z) = t exp(-z^2 + P(t)) with t = 1 / (1 + z/2).  Here P has degree 5
instead of 9.  It is the least-squares fit of ln(erfc(z) / t) + z^2 at 4000
Chebyshev nodes of t in [1/8, 1] (z in [0, 14]; beyond 14, exp(-z^2)
underflows binary32 anyway), turned into powers of t for Horner's rule.

Run it to print the binary32 coefficients (highest power first, as
zr_kernels.cuh uses them) and the largest error of ln erfc.  That error is
the relative error of erfc, measured on 400001 points with the binary32
Horner evaluation emulated.
"""
import numpy as np
from scipy.special import erfc

DEGREE = 5
T_MIN = 1.0 / 8.0


def target(t):
    z = 2.0 * (1.0 / t - 1.0)
    return np.log(erfc(z) / t) + z * z


def fit():
    n = 4000
    nodes = 0.5 * (1 + np.cos(np.pi * (np.arange(n) + 0.5) / n)) * (1 - T_MIN) + T_MIN
    cheb = np.polynomial.chebyshev.Chebyshev.fit(nodes, target(nodes), DEGREE)
    return cheb.convert(kind=np.polynomial.Polynomial).coef.astype(np.float32)


def horner32(coef, t):
    t32 = t.astype(np.float32)
    q = np.full_like(t32, coef[-1])
    for c in coef[-2::-1]:
        q = (q * t32 + c).astype(np.float32)
    return q


def main():
    coef = fit()
    t = np.linspace(T_MIN, 1.0, 400001)
    err = np.max(np.abs(horner32(coef, t).astype(np.float64) - target(t)))
    print("coefficients, highest power first:")
    print(", ".join(f"{c!r}" for c in (float(x) for x in coef[::-1])))
    print(f"max |error of ln erfc| on z in [0, 14]: {err:.3e} (2^{np.log2(err):.2f})")


if __name__ == "__main__":
    main()
