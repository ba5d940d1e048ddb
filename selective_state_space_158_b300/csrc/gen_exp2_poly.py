"""Generates the polynomial the fp32 path uses for 2^f on f in [-1/2, 1/2] (accurate exp2).

Method: Chebyshev interpolation (numpy.polynomial.chebyshev.chebinterpolate, in double
precision) of 2^f on [-1/2, 1/2], re-expanded in powers of f and rounded to float32. The kernel
reduces x to k + f with k = rint(x) (Cody and Waite's range reduction: f = x - k is exact in
fp32 for |x| < 2^22), evaluates p(f) by Horner's rule in fp32 and scales by 2^k through the
exponent field. This script reports the worst relative error of that fp32 evaluation on a dense
grid of f and the mean of the signed error (the evaluation must not be biased: decay factors
multiply into the state, and a consistently low or high factor would compound).
"""
import numpy as np
from numpy.polynomial import chebyshev as Ch
from numpy.polynomial import polynomial as P

DEGREE = 6


def coefficients(degree: int = DEGREE) -> np.ndarray:
    cu = Ch.cheb2poly(Ch.chebinterpolate(lambda u: np.exp2(u / 2.0), degree))  # u = 2 f
    ps = np.zeros(1)
    for k, a in enumerate(cu):
        ps = P.polyadd(ps, a * P.polypow([0.0, 2.0], k))
    return ps.astype(np.float32)


def evaluate(cf: np.ndarray, f: np.ndarray) -> np.ndarray:
    f = f.astype(np.float32)
    acc = np.full_like(f, cf[-1])
    for a in cf[-2::-1]:
        acc = (acc * f + a).astype(np.float32)  # numpy rounds each op to fp32 (no FMA)
    return acc


def errors(cf: np.ndarray):
    f = np.linspace(-0.5, 0.5, 1000001, dtype=np.float64).astype(np.float32)
    v = evaluate(cf, f).astype(np.float64)
    ref = np.exp2(f.astype(np.float64))
    rel = (v - ref) / ref
    return float(np.max(np.abs(rel))), float(np.mean(rel))


if __name__ == "__main__":
    cf = coefficients()
    print("// 2^f on [-1/2, 1/2], degree %d, low order first" % DEGREE)
    print(", ".join("%.9ef" % c for c in cf))
    mx, mean = errors(cf)
    print("// fp32 Horner (unfused): max relative error %.3g, mean signed %.3g" % (mx, mean))
