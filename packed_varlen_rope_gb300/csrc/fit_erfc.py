"""Coefficients of the erfc approximation used by the GeGLU kernels (csrc/glu.cu).

Form (the form of the Chebyshev-fitted erfc in Press et al., "Numerical Recipes",
section 6.2; the coefficients here are our own fit):

    erfc(z) = t * exp(-z^2 + P(t)),   t = 1 / (1 + z/2),   z >= 0,

where P is a polynomial in t.  The function F(t) = log(erfc(z) / t) + z^2 is smooth on
t in (0, 1] (z from infinity down to 0) and tends to log(1 / (2 sqrt(pi))) as t -> 0,
so a Chebyshev interpolant of F in t gives a small *relative* error of erfc everywhere.
F is evaluated with mpmath at 60 digits and interpolated at Chebyshev nodes.  Degree 9
leaves |P - F| < 2e-7; beyond it the binary32 evaluation in the kernel (the rounding
of -z^2 + P inside the exponential) dominates, so higher degrees buy nothing.  Run:
python fit_erfc.py [degree]  (prints the coefficients of P, highest degree first,
ready for a Horner evaluation, and the error of the fit).
"""
from __future__ import annotations

import mpmath
import numpy as np

mpmath.mp.dps = 60


def F(t: mpmath.mpf) -> mpmath.mpf:
    if t == 0:
        return mpmath.log(1 / (2 * mpmath.sqrt(mpmath.pi)))
    z = 2 * (1 / t - 1)
    return mpmath.log(mpmath.erfc(z) / t) + z * z


def fit(degree: int):
    # Chebyshev nodes on [0, 1]
    k = np.arange(degree + 1)
    x = np.cos((2 * k + 1) * np.pi / (2 * (degree + 1)))
    t = (x + 1) / 2
    y = np.array([float(F(mpmath.mpf(v))) for v in t])
    coef = np.polynomial.chebyshev.chebfit(x, y, degree)
    poly = np.polynomial.chebyshev.cheb2poly(coef)       # in x = 2t - 1
    # convert to a polynomial in t: x = 2t - 1
    p = np.polynomial.Polynomial(poly)
    pt = p(np.polynomial.Polynomial([-1.0, 2.0]))
    return pt.coef  # lowest degree first


def max_error(coef_t, n=20001):
    t = np.linspace(0.0, 1.0, n)
    approx = np.polynomial.polynomial.polyval(t, coef_t)
    exact = np.array([float(F(mpmath.mpf(v))) for v in t])
    return float(np.max(np.abs(approx - exact)))


if __name__ == "__main__":
    import sys

    degree = int(sys.argv[1]) if len(sys.argv) > 1 else 9
    c = fit(degree)
    print("degree %d: max |P - F| = %.3g on [0, 1]" % (degree, max_error(c, 20001)))
    print("coefficients, highest degree first:")
    for v in c[::-1]:
        print("    %.9ef," % v)
