"""Pins of the backward oracle (``oracle.mha_bwd``) against things other than
its own formulas: central finite differences of the (separately pinned)
forward oracle, closed forms and invariants of the gradients.

L = sum(out * dout); dq, dk, dv are dL/dq, dL/dk, dL/dv.
"""
import numpy as np
import pytest

import oracle
from oracle import MASK_CAUSAL, MASK_CAUSAL_TAIL, MASK_KEY_PADDING, MASK_QUERY_PADDING

C, KP, QP, TAIL = MASK_CAUSAL, MASK_KEY_PADDING, MASK_QUERY_PADDING, MASK_CAUSAL_TAIL


def _loss(q, k, v, dout, **kw):
    return float(np.sum(oracle.mha_fwd(q, k, v, **kw) * dout))


def _finite_differences(q, k, v, dout, eps=1e-5, **kw):
    grads = []
    for idx in range(3):
        args = [q.copy(), k.copy(), v.copy()]
        x = args[idx]
        g = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            mi = it.multi_index
            x0 = x[mi]
            x[mi] = x0 + eps
            lp = _loss(*args, dout, **kw)
            x[mi] = x0 - eps
            lm = _loss(*args, dout, **kw)
            x[mi] = x0
            g[mi] = (lp - lm) / (2 * eps)
        grads.append(g)
    return grads


CASES = [
    # B, H, Hkv, Lq, Lk, d, mask, lens, layout
    (1, 1, 1, 3, 4, 3, 0, None, "bhsd"),
    (2, 2, 2, 4, 4, 2, C, None, "bhsd"),
    (2, 2, 1, 3, 5, 2, KP, [2, 5], "bshd"),
    (2, 2, 2, 4, 4, 3, KP | QP, [0, 3], "bhsd"),
    (2, 4, 2, 2, 5, 2, TAIL | KP, [1, 4], "bshd"),
    (1, 2, 1, 5, 5, 2, C | KP, [3], "bhsd"),
    (2, 3, 3, 3, 6, 2, TAIL, None, "bhsd"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "m%d_%s_H%dKV%d" % (c[6], c[8], c[1], c[2]))
def test_gradients_match_finite_differences(case):
    B, H, Hkv, Lq, Lk, d, mask, lens, layout = case
    rng = np.random.default_rng(B * 100 + Lq * 10 + Lk + mask)
    qs, ks, os_ = ((B, Lq, H, d), (B, Lk, Hkv, d), (B, Lq, H, d)) if layout == "bshd" else \
        ((B, H, Lq, d), (B, Hkv, Lk, d), (B, H, Lq, d))
    q, k, v, dout = rng.normal(size=qs), rng.normal(size=ks), rng.normal(size=ks), \
        rng.normal(size=os_)
    kw = dict(mask_kind=mask, key_lengths=None if lens is None else np.array(lens, np.int32),
              scale=0.7, layout=layout)
    dq, dk, dv = oracle.mha_bwd(q, k, v, dout, **kw)
    fq, fk, fv = _finite_differences(q, k, v, dout, **kw)
    for got, want, name in ((dq, fq, "dq"), (dk, fk, "dk"), (dv, fv, "dv")):
        np.testing.assert_allclose(got, want, atol=2e-8, rtol=1e-6, err_msg=name)


def test_single_key():
    # one key: every allowed row's output is that value row; dq = dk = 0 and
    # dv_0 = the sum of dout over the rows
    rng = np.random.default_rng(1)
    q, k, v = rng.normal(size=(2, 3, 4, 5)), rng.normal(size=(2, 3, 1, 5)), \
        rng.normal(size=(2, 3, 1, 5))
    dout = rng.normal(size=(2, 3, 4, 5))
    dq, dk, dv = oracle.mha_bwd(q, k, v, dout, scale=0.3)
    assert np.all(dq == 0) and np.all(dk == 0)
    np.testing.assert_allclose(dv[:, :, 0], dout.sum(axis=2), rtol=1e-14, atol=1e-14)


def test_zero_scale():
    # scale 0: uniform weights over the allowed keys; dq = dk = 0 and
    # dv_j = sum over the rows that allow j of dout_i / |A_i|
    rng = np.random.default_rng(2)
    L, d = 6, 3
    q, k, v, dout = (rng.normal(size=(1, 2, L, d)) for _ in range(4))
    dq, dk, dv = oracle.mha_bwd(q, k, v, dout, mask_kind=C, scale=0.0)
    assert np.all(dq == 0) and np.all(dk == 0)
    want = np.zeros_like(v)
    for i in range(L):
        want[:, :, : i + 1] += dout[:, :, i : i + 1] / (i + 1)
    np.testing.assert_allclose(dv, want, rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("mask,lens", [(0, None), (C, None), (KP | QP, [3, 7])])
def test_key_gradients_sum_to_zero_and_shift_invariance(mask, lens):
    # sum_j dL/ds_ij = 0 for every row, so the key gradients of a head sum to
    # zero, and shifting every key by one vector changes no gradient
    rng = np.random.default_rng(3)
    q, k, v, dout = (rng.normal(size=(2, 2, 7, 4)) for _ in range(4))
    kw = dict(mask_kind=mask, key_lengths=None if lens is None else np.array(lens, np.int32),
              scale=0.5)
    dq, dk, dv = oracle.mha_bwd(q, k, v, dout, **kw)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-13)
    c = rng.normal(size=(1, 1, 1, 4))
    dq2, dk2, dv2 = oracle.mha_bwd(q, k + c, v, dout, **kw)
    for a, b in ((dq, dq2), (dk, dk2), (dv, dv2)):
        np.testing.assert_allclose(a, b, atol=1e-12)


def test_padded_rows_and_keys_get_nothing():
    # query-padding rows have a fixed output: zero dq; keys past the length
    # are never read: zero dk, dv
    rng = np.random.default_rng(4)
    q, k, v, dout = (rng.normal(size=(2, 2, 6, 3)) for _ in range(4))
    lens = np.array([4, 0], np.int32)
    dq, dk, dv = oracle.mha_bwd(q, k, v, dout, mask_kind=KP | QP, key_lengths=lens, scale=0.5)
    assert np.all(dq[0, :, 4:] == 0) and np.all(dq[1] == 0)
    assert np.all(dk[0, :, 4:] == 0) and np.all(dv[0, :, 4:] == 0)
    assert np.all(dk[1] == 0) and np.all(dv[1] == 0)


def test_grouped_heads_sum_over_their_query_heads():
    rng = np.random.default_rng(5)
    B, H, Hkv, L, d = 2, 6, 2, 5, 3
    q, dout = rng.normal(size=(B, H, L, d)), rng.normal(size=(B, H, L, d))
    k, v = rng.normal(size=(B, Hkv, L, d)), rng.normal(size=(B, Hkv, L, d))
    g = H // Hkv
    dq, dk, dv = oracle.mha_bwd(q, k, v, dout, mask_kind=C, scale=0.4)
    rq, rk, rv = oracle.mha_bwd(q, np.repeat(k, g, axis=1), np.repeat(v, g, axis=1), dout,
                                mask_kind=C, scale=0.4)
    np.testing.assert_allclose(dq, rq, atol=1e-13)
    np.testing.assert_allclose(dk, rk.reshape(B, Hkv, g, L, d).sum(axis=2), atol=1e-13)
    np.testing.assert_allclose(dv, rv.reshape(B, Hkv, g, L, d).sum(axis=2), atol=1e-13)


def test_bshd_layout_equals_bhsd():
    rng = np.random.default_rng(6)
    q, dout = rng.normal(size=(2, 4, 5, 3)), rng.normal(size=(2, 4, 5, 3))
    k, v = rng.normal(size=(2, 2, 7, 3)), rng.normal(size=(2, 2, 7, 3))
    lens = np.array([7, 3], np.int32)
    a = oracle.mha_bwd(q, k, v, dout, mask_kind=KP, key_lengths=lens, scale=0.5)
    t = lambda x: np.ascontiguousarray(x.transpose(0, 2, 1, 3))
    b = oracle.mha_bwd(t(q), t(k), t(v), t(dout), mask_kind=KP, key_lengths=lens, scale=0.5,
                       layout="bshd")
    for x, y in zip(a, b):
        np.testing.assert_array_equal(t(y), x)


def test_units_and_row_ranges():
    # a subset of units gives those units' gradients; row ranges split the sums
    rng = np.random.default_rng(7)
    q, k, v, dout = (rng.normal(size=(3, 2, 6, 3)) for _ in range(4))
    full = oracle.mha_bwd(q, k, v, dout, mask_kind=C, scale=0.5)
    part = oracle.mha_bwd(q, k, v, dout, mask_kind=C, scale=0.5, units=[4, 1])
    for f, p in zip(full, part):
        np.testing.assert_array_equal(p[2, 0], f[2, 0])
        np.testing.assert_array_equal(p[0, 1], f[0, 1])
        assert np.all(p[1] == 0) and np.all(p[0, 0] == 0)
    lo = oracle.mha_bwd(q, k, v, dout, mask_kind=C, scale=0.5, rows=(0, 2))
    hi = oracle.mha_bwd(q, k, v, dout, mask_kind=C, scale=0.5, rows=(2, 6))
    for f, a, b in zip(full, lo, hi):
        np.testing.assert_allclose(a + b, f, atol=1e-13)


def test_bf16_inputs_widen_exactly():
    import gen
    rng = np.random.default_rng(8)
    xs = [gen.f64_to_bf16_bits(rng.normal(size=(1, 2, 5, 4))) for _ in range(4)]
    a = oracle.mha_bwd(*xs, mask_kind=C, scale=0.5)
    b = oracle.mha_bwd(*[gen.bf16_bits_to_f64(x) for x in xs], mask_kind=C, scale=0.5)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_rejects_bad_arguments():
    z = np.zeros((1, 2, 3, 4))
    with pytest.raises(ValueError):
        oracle.mha_bwd(z, z, z, z, mask_kind=KP, scale=1.0)  # lengths missing
    with pytest.raises(ValueError):
        oracle.mha_bwd(z, np.zeros((1, 2, 4, 4)), np.zeros((1, 2, 4, 4)), z, mask_kind=C,
                       scale=1.0)  # causal with Lq != Lk
    with pytest.raises(ValueError):
        oracle.mha_bwd(z, z, z, np.zeros((1, 2, 3, 5)), scale=1.0)  # dout shape
