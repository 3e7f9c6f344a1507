"""The cubic that the long-sequence kernel evaluates on the FMA pipes for part
of its exponentials (exp2_poly2 in csrc/ptx.cuh): its coefficients are the
minimax fit that fit_exp2_poly.py derives, and its float32 evaluation, with
the kernel's range reduction and exponent add, stays within the stated
relative error bound against exp2 in float64."""
import os
import re
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "transformer_head_scaled_mha_gb300")


def header_coefficients():
    src = open(os.path.join(PKG, "csrc", "ptx.cuh")).read()
    return [float(re.search(r"kExp2C%d = ([-+0-9.e]+)f;" % i, src).group(1)) for i in range(4)]


@pytest.fixture(scope="module")
def fit():
    pytest.importorskip("scipy")
    sys.path.insert(0, PKG)
    try:
        import fit_exp2_poly
    finally:
        sys.path.remove(PKG)
    return fit_exp2_poly


def test_header_holds_the_fitted_coefficients(fit):
    c, err = fit.fit()
    assert err < 7.5e-5
    assert header_coefficients() == pytest.approx([float(np.float32(v)) for v in c], rel=1e-8)


def test_float32_evaluation_within_bound(fit):
    c = header_coefficients()
    x = np.linspace(-125.0, 8.0, 1_000_001).astype(np.float32)
    got = fit.eval_f32(x, c).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    assert np.max(np.abs(got - ref) / ref) < 7.6e-5
    # below the clamp the result is tiny and positive, never negative or NaN
    lo = fit.eval_f32(np.array([-126.0, -200.0, -1e30], dtype=np.float32), c)
    assert np.all(np.isfinite(lo)) and np.all(lo >= 0) and np.all(lo < 2.0 ** -125)


def test_range_reduction_splits_exactly(fit):
    # x = n + f with n = round-half-even(x): integers give f = 0, so 2^n
    # scaled by p(0) (relative error of p alone)
    c = header_coefficients()
    x = np.arange(-120, 9, dtype=np.float32)
    got = fit.eval_f32(x, c).astype(np.float64)
    assert np.allclose(got / np.exp2(x.astype(np.float64)), c[0], rtol=0, atol=1e-7)
