"""Derives the cubic that the long-sequence kernel uses for part of its
exponentials (2^x on the FMA pipes instead of the MUFU unit).

Method (range reduction as in Cody and Waite, "Software Manual for the
Elementary Functions", 1980, specialised to base 2, where it is exact):
2^x = 2^n * 2^f with n = round(x) and f = x - n in [-1/2, 1/2]; 2^f is
replaced by the cubic p(f) that minimises the largest RELATIVE error on
[-1/2, 1/2] (a minimax fit, solved here as a linear programme over a dense
grid), and 2^n is applied by adding n to the exponent field of p(f).

Running this file prints the float32 coefficients written in ptx.cuh
(kExp2C0..kExp2C3) and the relative error bound of the float32 evaluation.
"""
import numpy as np
from scipy.optimize import linprog


def fit(degree=3, n=4001):
    f = np.linspace(-0.5, 0.5, n)
    y = np.exp2(f)
    V = np.vander(f, degree + 1, increasing=True)  # columns f^0 .. f^degree
    # minimise t subject to |(V c - y) / y| <= t
    A = np.vstack([np.hstack([V / y[:, None], -np.ones((n, 1))]),
                   np.hstack([-V / y[:, None], -np.ones((n, 1))])])
    b = np.concatenate([np.ones(n), -np.ones(n)])
    cost = np.zeros(degree + 2)
    cost[-1] = 1.0
    res = linprog(cost, A_ub=A, b_ub=b, bounds=[(None, None)] * (degree + 2), method="highs")
    assert res.success
    return res.x[:-1], res.x[-1]


def eval_f32(x, c):
    """The kernel's float32 steps, emulated: clamp, round by the 1.5 * 2^23
    shift, Horner in float32 (fused multiply-adds rounded once), exponent add."""
    x = np.maximum(np.asarray(x, dtype=np.float32), np.float32(-126.0))
    magic = np.float32(12582912.0)
    t = (x + magic).astype(np.float32)
    n = (t - magic).astype(np.float32)
    f = (x - n).astype(np.float32)
    c = [np.float32(v) for v in c]
    p = ((c[3].astype(np.float64) * f + c[2]).astype(np.float32))
    p = ((p.astype(np.float64) * f + c[1]).astype(np.float32))
    p = ((p.astype(np.float64) * f + c[0]).astype(np.float32))
    bits = p.view(np.uint32).astype(np.int64) + (n.astype(np.int64) << 23)
    return (bits & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


if __name__ == "__main__":
    c, t = fit()
    c32 = [float(np.float32(v)) for v in c]
    print("minimax relative error of the real-coefficient cubic: %.3e" % t)
    for i, v in enumerate(c32):
        print("kExp2C%d = %.9ef  (%s)" % (i, v, np.float32(v).view(np.uint32)))
    x = np.linspace(-126.0, 8.0, 2_000_001, dtype=np.float64).astype(np.float32)
    got = eval_f32(x, c32).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    print("float32 evaluation on [-126, 8]: max relative error %.3e" %
          float(np.max(np.abs(got - ref) / ref)))
