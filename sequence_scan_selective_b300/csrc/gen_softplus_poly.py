"""Derive the polynomial used by the kernels' softplus.

softplus(x) = max(x, 0) + log1p(e) with e = exp(-|x|) in (0, 1].  log1p(e) = e * P(e), where P is
the degree-6 Chebyshev interpolant of log1p(e)/e on [0, 1], rewritten in the monomial basis and
rounded to fp32.  Run this script to print the coefficients (lowest order first) and the fp32
Horner error against numpy's log1p.
"""
import numpy as np
from numpy.polynomial import chebyshev as Ch
from numpy.polynomial import polynomial as Po

DEG = 6


def coefficients(deg=DEG):
    f = lambda e: np.where(e == 0, 1.0, np.log1p(e) / np.where(e == 0, 1.0, e))
    c = Ch.chebinterpolate(lambda t: f((t + 1) / 2), deg)       # t = 2e - 1 in [-1, 1]
    p_t = Ch.cheb2poly(c)
    return Po.Polynomial(p_t)(Po.Polynomial([-1.0, 2.0])).coef    # in powers of e


def horner_f32(coef, e):
    c32 = np.asarray(coef, np.float32)
    e32 = np.asarray(e, np.float32)
    acc = np.full_like(e32, c32[-1])
    for k in range(len(c32) - 2, -1, -1):
        acc = (acc * e32 + c32[k]).astype(np.float32)
    return (acc * e32).astype(np.float32)


if __name__ == "__main__":
    co = coefficients()
    for k, v in enumerate(co):
        print(f"c{k} = {np.float32(v)!r}  ({float(np.float32(v)).hex()})")
    e = np.linspace(0, 1, 400001)[1:]
    print("max rel err (fp32 Horner):", float(np.max(np.abs(horner_f32(co, e) - np.log1p(e)) / np.log1p(e))))
