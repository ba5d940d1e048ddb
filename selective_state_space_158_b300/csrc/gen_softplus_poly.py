"""Generates the polynomial the kernels use for log1p(s) on s in [0, 1].

Method: Chebyshev interpolation (numpy.polynomial.chebyshev.chebinterpolate, degree 9, in
double precision) of f(s) = log1p(s) / s on [0, 1], re-expanded in powers of s and rounded to
float32. The kernel evaluates log1p(s) = s * p(s) by Horner's rule in fp32; this script also
reports the fp32 evaluation's worst relative error on a dense grid (about 1.6e-7).

softplus(x) = max(x, 0) + log1p(exp(-|x|)) then needs one SFU exponential and this polynomial.
"""
import numpy as np
from numpy.polynomial import chebyshev as Ch
from numpy.polynomial import polynomial as P

DEGREE = 9


def coefficients(degree: int = DEGREE) -> np.ndarray:
    def f(u):
        s = (u + 1.0) / 2.0
        out = np.ones_like(s)
        nz = s != 0
        out[nz] = np.log1p(s[nz]) / s[nz]
        return out

    cu = Ch.cheb2poly(Ch.chebinterpolate(f, degree))  # power series in u = 2s - 1
    ps = np.zeros(1)
    for k, a in enumerate(cu):
        ps = P.polyadd(ps, a * P.polypow([-1.0, 2.0], k))
    return ps.astype(np.float32)


def max_rel_error(cf: np.ndarray) -> float:
    s = np.linspace(0.0, 1.0, 400001, dtype=np.float64)[1:].astype(np.float32)
    acc = np.full_like(s, cf[-1])
    for a in cf[-2::-1]:
        acc = (acc * s + a).astype(np.float32)
    v = (s * acc).astype(np.float64)
    ref = np.log1p(s.astype(np.float64))
    return float(np.max(np.abs(v - ref) / ref))


if __name__ == "__main__":
    cf = coefficients()
    print("// log1p(s)/s on [0,1], degree %d, low order first" % DEGREE)
    print(", ".join("%.9ef" % c for c in cf))
    print("// max relative error of s*p(s) in fp32: %.3g" % max_rel_error(cf))
