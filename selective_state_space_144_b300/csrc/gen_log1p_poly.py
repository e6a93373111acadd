"""Generate the polynomial used by the kernels' softplus for log1p on [0, 1].

log1p(e) = e * P(s), s = 2e - 1, where P interpolates log1p(e)/e at the
degree+1 Chebyshev nodes of [0, 1].  Evaluated by Horner in fp32 the result
has a maximum relative error of about 1.9e-7 over [0, 1] for degree 8 (this
script prints it).  Run:  python gen_log1p_poly.py [degree]
"""
import sys

import numpy as np
from numpy.polynomial import chebyshev as cheb


def ratio(e):
    e = np.asarray(e, dtype=np.float64)
    out = np.ones_like(e)
    m = e > 0
    out[m] = np.log1p(e[m]) / e[m]
    return out


def fit(deg):
    k = np.arange(deg + 1)
    nodes = 0.5 + 0.5 * np.cos(np.pi * (k + 0.5) / (deg + 1))
    c = cheb.chebfit(2 * nodes - 1, ratio(nodes), deg)
    return cheb.cheb2poly(c)          # monomial coefficients in s, low first


def fp32_max_rel_err(p):
    xs = np.linspace(0.0, 1.0, 200001)
    s = (2 * xs - 1).astype(np.float32)
    acc = np.float32(p[-1])
    for a in p[-2::-1]:
        acc = (acc * s + np.float32(a)).astype(np.float32)
    approx = (xs.astype(np.float32) * acc).astype(np.float64)
    ref = np.log1p(xs)
    rel = np.abs(approx - ref)[1:] / ref[1:]
    return float(rel.max())


if __name__ == "__main__":
    deg = int(sys.argv[1]) if len(sys.argv) > 1 else 8
    p = fit(deg)
    print(f"// degree {deg}, fp32 max rel err {fp32_max_rel_err(p):.3e}")
    for i, a in enumerate(p):
        print(f"constexpr float kLog1pP{i} = {np.float32(a)!r}f;".replace(
            "np.float32(", "").replace(")f", "f"))
