"""Pins for the fp64 oracle, before any GPU code is trusted against it.

Each test fixes the oracle to something other than itself: numbers the pages
print, closed forms, invariants the pages state, the variance argument for
the 1/sqrt(d_k) scale, and a 50-digit brute force on tiny inputs.  A plausible
slip in the oracle (a dropped term, a sign, a swapped operand, a wrong mask
index, softmax over the wrong axis) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import gen
import oracle
from oracle import MASK_CAUSAL, MASK_KEY_PADDING, MASK_QUERY_PADDING

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")


def _scale(text):
    return {"1/sqrt(2)": 1.0 / math.sqrt(2.0), "1": 1.0}[text]


# --------------------------------------------------------------------------
# printed values: the three-token worked example and its two variants
# --------------------------------------------------------------------------
@pytest.mark.parametrize("case", ["scaled_identity", "unscaled_identity", "was_doubled"])
def test_worked_example(oracle_lib, case):
    g = json.load(open(GOLDEN))
    c = g["cases"][case]
    tol = 0.5 * 10.0 ** -g["decimals"] + 1e-12
    X = np.array(c["X"], dtype=np.float64)[None, None]
    out, w, s = oracle.mha_fwd(X, X, X, scale=_scale(c["scale"]), return_weights=True,
                               return_scores=True)
    for row, vals in c.get("out", {}).items():
        np.testing.assert_allclose(out[0, 0, int(row)], vals, rtol=0, atol=tol)
    for row, vals in c.get("weights", {}).items():
        np.testing.assert_allclose(w[0, 0, int(row)], vals, rtol=0, atol=tol)
    for row, vals in c.get("scores", {}).items():
        np.testing.assert_allclose(s[0, 0, int(row)], vals, rtol=0, atol=tol)


# --------------------------------------------------------------------------
# invariants and closed forms
# --------------------------------------------------------------------------
def _rand(B, H, Lq, Lk, dk, dv, seed=7):
    q = gen.tensor(seed, 0, (B, H, Lq, dk), "f64")
    k = gen.tensor(seed, 1, (B, H, Lk, dk), "f64")
    v = gen.tensor(seed, 2, (B, H, Lk, dv), "f64")
    return q, k, v


MASKS = [
    (0, None),
    (MASK_CAUSAL, None),
    (MASK_KEY_PADDING, [3, 9, 0, 1]),
    (MASK_KEY_PADDING | MASK_QUERY_PADDING, [3, 9, 0, 1]),
    (MASK_KEY_PADDING | MASK_CAUSAL, [4, 9, 0, 2]),
]


@pytest.mark.parametrize("mask,lens", MASKS)
def test_rows_sum_to_one_and_masked_weights_zero(oracle_lib, mask, lens):
    B, H, L, d = 4, 3, 9, 5
    q, k, v = _rand(B, H, L, L, d, d)
    out, w = oracle.mha_fwd(q, k, v, mask_kind=mask, key_lengths=lens, scale=0.4,
                            return_weights=True)
    for b in range(B):
        lb = L if lens is None else max(0, min(lens[b], L))
        for i in range(L):
            allowed = np.ones(L, bool)
            if mask & MASK_CAUSAL:
                allowed &= np.arange(L) <= i
            if mask & MASK_KEY_PADDING:
                allowed &= np.arange(L) < lb
            qpad = bool(mask & MASK_QUERY_PADDING) and i >= lb
            rs = w[b, :, i].sum(axis=-1)
            if qpad or not allowed.any():
                assert np.all(w[b, :, i] == 0.0)
                assert np.all(out[b, :, i] == 0.0) and not np.any(np.signbit(out[b, :, i]))
            else:
                np.testing.assert_allclose(rs, 1.0, rtol=0, atol=1e-14)
                assert np.all(w[b, :, i][:, ~allowed] == 0.0)
                assert np.all(w[b, :, i][:, allowed] > 0.0)


@pytest.mark.parametrize("mask,lens", MASKS)
def test_zero_query_gives_mean_of_allowed_values(oracle_lib, mask, lens):
    # Q = 0 makes every allowed score equal, so the softmax is uniform over the
    # allowed keys and the output is the plain mean of their value rows.
    B, H, L, d = 4, 2, 7, 3
    _, k, v = _rand(B, H, L, L, d, d)
    q = np.zeros_like(k)
    out = oracle.mha_fwd(q, k, v, mask_kind=mask, key_lengths=lens, scale=0.125)
    for b in range(B):
        lb = L if lens is None else max(0, min(lens[b], L))
        for i in range(L):
            hi = L
            if mask & MASK_KEY_PADDING:
                hi = min(hi, lb)
            if mask & MASK_CAUSAL:
                hi = min(hi, i + 1)
            if (mask & MASK_QUERY_PADDING and i >= lb) or hi == 0:
                expect = np.zeros((H, d))
            else:
                expect = v[b, :, :hi].mean(axis=1)
            np.testing.assert_allclose(out[b, :, i], expect, rtol=0, atol=1e-14)


def test_zero_scale_gives_mean_of_values(oracle_lib):
    q, k, v = _rand(2, 2, 5, 6, 4, 3)
    out = oracle.mha_fwd(q, k, v, scale=0.0)
    np.testing.assert_allclose(out, np.broadcast_to(v.mean(axis=2, keepdims=True), out.shape),
                               rtol=0, atol=1e-14)


def test_causal_row_zero_is_first_value(oracle_lib):
    q, k, v = _rand(2, 3, 11, 11, 8, 6)
    out = oracle.mha_fwd(q, k, v, mask_kind=MASK_CAUSAL, scale=0.35)
    np.testing.assert_array_equal(out[:, :, 0], v[:, :, 0])


def test_single_key_gives_its_value(oracle_lib):
    q, k, v = _rand(2, 2, 5, 1, 4, 3)
    out = oracle.mha_fwd(q, k, v, scale=0.5)
    np.testing.assert_array_equal(out, np.broadcast_to(v[:, :, :1], out.shape))
    # the same through key padding with length 1
    q, k, v = _rand(2, 2, 5, 5, 4, 3)
    out = oracle.mha_fwd(q, k, v, mask_kind=MASK_KEY_PADDING, key_lengths=[1, 1], scale=0.5)
    np.testing.assert_array_equal(out, np.broadcast_to(v[:, :, :1], out.shape))


def test_lengths_are_clamped(oracle_lib):
    q, k, v = _rand(3, 1, 4, 4, 2, 2)
    a = oracle.mha_fwd(q, k, v, mask_kind=MASK_KEY_PADDING | MASK_QUERY_PADDING,
                       key_lengths=[-5, 99, 4], scale=1.0)
    b = oracle.mha_fwd(q, k, v, mask_kind=MASK_KEY_PADDING | MASK_QUERY_PADDING,
                       key_lengths=[0, 4, 4], scale=1.0)
    np.testing.assert_array_equal(a, b)
    assert np.all(a[0] == 0.0)


def test_sqrt_dk_scaling_statistics():
    # Variance of a dot product of two d_k-vectors with i.i.d. unit-variance
    # entries is d_k; the pages' own run over 4,000 pairs printed standard
    # deviations 1.99 / 7.89 / 22.54 for d_k = 4 / 64 / 512 and about 1 after
    # dividing by sqrt(d_k) (aicassindra.com, "Why the dot product is divided
    # by the square root of d_k").  Checked here on the generator's N(0,1)
    # streams through the oracle's scaled logits.
    printed = {4: 1.99, 64: 7.89, 512: 22.54}
    n = 4000
    for dk, page_std in printed.items():
        q = gen.tensor(11, 0, (n, 1, 1, dk), "f64")
        k = gen.tensor(11, 1, (n, 1, 1, dk), "f64")
        v = np.zeros((n, 1, 1, 1))
        _, raw = oracle.mha_fwd(q, k, v, scale=1.0, return_scores=True)
        _, scaled = oracle.mha_fwd(q, k, v, scale=1.0 / math.sqrt(dk), return_scores=True)
        sd_raw = raw.reshape(-1).std()
        sd_scaled = scaled.reshape(-1).std()
        assert abs(sd_raw / math.sqrt(dk) - 1.0) < 0.05
        assert abs(sd_raw / page_std - 1.0) < 0.05
        assert abs(sd_scaled - 1.0) < 0.05


def test_query_permutation_permutes_rows_exactly(oracle_lib):
    q, k, v = _rand(1, 2, 9, 7, 4, 3)
    perm = np.array([4, 0, 8, 2, 6, 1, 7, 3, 5])
    a = oracle.mha_fwd(q, k, v, scale=0.6)
    b = oracle.mha_fwd(q[:, :, perm], k, v, scale=0.6)
    np.testing.assert_array_equal(b, a[:, :, perm])


def test_key_value_permutation_leaves_output(oracle_lib):
    q, k, v = _rand(1, 2, 6, 8, 4, 3)
    perm = np.array([3, 7, 0, 5, 1, 6, 2, 4])
    a = oracle.mha_fwd(q, k, v, scale=0.6)
    b = oracle.mha_fwd(q, k[:, :, perm], v[:, :, perm], scale=0.6)
    np.testing.assert_allclose(b, a, rtol=0, atol=1e-14)


def test_value_affine_maps(oracle_lib):
    # Weights sum to one, so adding c to every value row adds c to the output,
    # and the output is linear in V: out(V A) = out(V) A.
    q, k, v = _rand(2, 2, 5, 6, 4, 3)
    c = np.array([0.5, -2.0, 3.25])
    A = np.array([[1.0, 2.0], [-1.0, 0.5], [0.25, 3.0]])
    base = oracle.mha_fwd(q, k, v, scale=0.3)
    np.testing.assert_allclose(oracle.mha_fwd(q, k, v + c, scale=0.3), base + c, atol=1e-13)
    np.testing.assert_allclose(oracle.mha_fwd(q, k, v @ A, scale=0.3), base @ A, atol=1e-13)


def test_shifting_all_keys_changes_nothing(oracle_lib):
    # k_j -> k_j + u adds scale*q.u to every score of a row: a per-row constant
    # that softmax removes.
    q, k, v = _rand(2, 2, 5, 6, 4, 3)
    u = np.array([0.3, -1.2, 2.0, 0.7])
    a = oracle.mha_fwd(q, k, v, scale=0.4)
    b = oracle.mha_fwd(q, k + u, v, scale=0.4)
    np.testing.assert_allclose(b, a, rtol=0, atol=1e-13)


def test_future_tokens_never_change_earlier_rows(oracle_lib):
    # "Test that changing a future token never changes an earlier output"
    # (aicassindra.com, "Pitfalls when reproducing the paper").
    L = 10
    q, k, v = _rand(1, 2, L, L, 4, 3)
    base = oracle.mha_fwd(q, k, v, mask_kind=MASK_CAUSAL, scale=0.5)
    for t in range(L):
        k2, v2 = k.copy(), v.copy()
        k2[:, :, t] += 7.0
        v2[:, :, t] -= 3.0
        out = oracle.mha_fwd(q, k2, v2, mask_kind=MASK_CAUSAL, scale=0.5)
        np.testing.assert_array_equal(out[:, :, :t], base[:, :, :t])
        if t < L:
            assert not np.array_equal(out[:, :, t:], base[:, :, t:])


def test_padded_keys_never_matter(oracle_lib):
    L = 8
    lens = [5, 2]
    q, k, v = _rand(2, 2, L, L, 4, 3)
    base = oracle.mha_fwd(q, k, v, mask_kind=MASK_KEY_PADDING, key_lengths=lens, scale=0.5)
    k2, v2 = k.copy(), v.copy()
    for b, lb in enumerate(lens):
        k2[b, :, lb:] = 1e3
        v2[b, :, lb:] = -1e3
    out = oracle.mha_fwd(q, k2, v2, mask_kind=MASK_KEY_PADDING, key_lengths=lens, scale=0.5)
    np.testing.assert_array_equal(out, base)


def test_heads_and_batches_are_independent(oracle_lib):
    q, k, v = _rand(3, 4, 5, 6, 4, 3)
    lens = [2, 6, 4]
    m = MASK_KEY_PADDING
    a = oracle.mha_fwd(q, k, v, mask_kind=m, key_lengths=lens, scale=0.7)
    hp = np.array([2, 0, 3, 1])
    b = oracle.mha_fwd(q[:, hp], k[:, hp], v[:, hp], mask_kind=m, key_lengths=lens, scale=0.7)
    np.testing.assert_array_equal(b, a[:, hp])
    bp = np.array([1, 2, 0])
    c = oracle.mha_fwd(q[bp], k[bp], v[bp], mask_kind=m, key_lengths=np.array(lens)[bp],
                       scale=0.7)
    np.testing.assert_array_equal(c, a[bp])


def test_row_subset_matches_full(oracle_lib):
    q, k, v = _rand(2, 3, 7, 7, 4, 5)
    full = oracle.mha_fwd(q, k, v, mask_kind=MASK_CAUSAL, scale=0.3)
    rows = np.array([0, 5, 13, 20, 41])
    sub = oracle.mha_fwd(q, k, v, mask_kind=MASK_CAUSAL, scale=0.3, rows=rows)
    np.testing.assert_array_equal(sub, full.reshape(-1, 5)[rows])


def test_stored_types_widen_exactly(oracle_lib):
    spec = dict(B=2, H=2, Lq=6, Lk=6, dk=4, dv=4, dtype="bf16", amp=1.0)
    q, k, v, _ = gen.make_inputs(spec, seed=3)
    a = oracle.mha_fwd(q, k, v, scale=0.5)
    b = oracle.mha_fwd(gen.as_f64(q, "bf16"), gen.as_f64(k, "bf16"), gen.as_f64(v, "bf16"),
                       scale=0.5)
    np.testing.assert_array_equal(a, b)
    q32 = gen.tensor(3, 0, (2, 2, 6, 4), "f32")
    c = oracle.mha_fwd(q32, q32, q32, scale=0.5)
    d = oracle.mha_fwd(q32.astype(np.float64), q32.astype(np.float64), q32.astype(np.float64),
                       scale=0.5)
    np.testing.assert_array_equal(c, d)


def test_rejects_bad_arguments(oracle_lib):
    q, k, v = _rand(1, 1, 4, 5, 2, 2)
    with pytest.raises(ValueError):
        oracle.mha_fwd(q, k, v, mask_kind=MASK_CAUSAL, scale=1.0)  # causal needs Lq == Lk
    with pytest.raises(ValueError):
        oracle.mha_fwd(q, k, v, mask_kind=MASK_KEY_PADDING, scale=1.0)  # lengths missing


def test_empty_shapes(oracle_lib):
    q, k, v = _rand(2, 2, 0, 5, 3, 3)
    assert oracle.mha_fwd(q, k, v, scale=1.0).shape == (2, 2, 0, 3)
    q, k, v = _rand(2, 2, 3, 0, 3, 3)
    out = oracle.mha_fwd(q, k, v, scale=1.0)
    assert out.shape == (2, 2, 3, 3) and np.all(out == 0.0)


# --------------------------------------------------------------------------
# brute force at 50 significant digits, straight from the definition
# softmax(QK^T * scale) V with masked logits at -inf (no max subtraction)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("mask,lens", [(0, None), (MASK_CAUSAL, None),
                                       (MASK_KEY_PADDING | MASK_QUERY_PADDING, [2, 5]),
                                       (MASK_KEY_PADDING, [0, 3]),
                                       (8 | MASK_KEY_PADDING, [4, 2]), (8, None)])
def test_brute_force_high_precision(oracle_lib, mask, lens):
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    B, H, L, dk, dv = 2, 2, 5, 3, 2
    q, k, v = _rand(B, H, L, L, dk, dv, seed=21)
    scale = 0.61
    out = oracle.mha_fwd(q, k, v, mask_kind=mask, key_lengths=lens, scale=scale)
    for b in range(B):
        lb = L if lens is None else lens[b]
        for h in range(H):
            for i in range(L):
                logits = []
                for j in range(L):
                    masked = ((mask & MASK_CAUSAL and j > i) or (mask & MASK_KEY_PADDING and j >= lb)
                              or (mask & 8 and j > lb - L + i))
                    if masked:
                        logits.append(None)
                    else:
                        dot = mp.fsum(mp.mpf(q[b, h, i, c]) * mp.mpf(k[b, h, j, c])
                                      for c in range(dk))
                        logits.append(mp.mpf(scale) * dot)
                e = [mp.e ** x if x is not None else mp.mpf(0) for x in logits]
                z = mp.fsum(e)
                qpad = mask & MASK_QUERY_PADDING and i >= lb
                for c in range(dv):
                    if qpad or z == 0:
                        ref = mp.mpf(0)
                    else:
                        ref = mp.fsum(e[j] * mp.mpf(v[b, h, j, c]) for j in range(L)) / z
                    assert abs(float(ref) - out[b, h, i, c]) < 1e-14


# --------------------------------------------------------------------------
# grouped key/value heads and the [B, L, H, d] layout, pinned to the
# multi-head oracle above
# --------------------------------------------------------------------------
@pytest.mark.parametrize("mask,lens", MASKS)
@pytest.mark.parametrize("H,Hkv", [(4, 4), (4, 2), (6, 1), (6, 3)])
def test_grouped_heads_equal_repeated_heads(oracle_lib, mask, lens, H, Hkv):
    # Sharing key/value head g among H/Hkv query heads is multi-head attention
    # with that head repeated (zeroshotmind.com, "Many heads, many subspaces").
    B, L, d = 4, 9, 5
    q = gen.tensor(3, 0, (B, H, L, d), "f64")
    k = gen.tensor(3, 1, (B, Hkv, L, d), "f64")
    v = gen.tensor(3, 2, (B, Hkv, L, d), "f64")
    got = oracle.mha_fwd(q, k, v, mask_kind=mask, key_lengths=lens, scale=0.45)
    rep = H // Hkv
    ref = oracle.mha_fwd(q, np.repeat(k, rep, axis=1), np.repeat(v, rep, axis=1),
                         mask_kind=mask, key_lengths=lens, scale=0.45)
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("mask,lens", MASKS)
def test_bshd_layout_equals_bhsd(oracle_lib, mask, lens):
    # the layout before the head split, [B, L, h, d_k] (aicassindra.com, "A
    # faithful layer in code"), holds the same numbers as [B, h, L, d_k]
    B, H, Hkv, L, d = 4, 4, 2, 9, 5
    q = gen.tensor(4, 0, (B, H, L, d), "f64")
    k = gen.tensor(4, 1, (B, Hkv, L, d), "f64")
    v = gen.tensor(4, 2, (B, Hkv, L, d), "f64")
    ref = oracle.mha_fwd(q, k, v, mask_kind=mask, key_lengths=lens, scale=0.3)
    t = lambda a: np.ascontiguousarray(a.transpose(0, 2, 1, 3))
    got = oracle.mha_fwd(t(q), t(k), t(v), mask_kind=mask, key_lengths=lens, scale=0.3,
                         layout="bshd")
    np.testing.assert_array_equal(got, t(ref))
    rows = np.array([0, 7, 20, 35, 143])
    np.testing.assert_array_equal(
        oracle.mha_fwd(t(q), t(k), t(v), mask_kind=mask, key_lengths=lens, scale=0.3,
                       layout="bshd", rows=rows), ref.reshape(-1, d)[rows])


def test_grouped_heads_reject_non_divisor(oracle_lib):
    q = np.zeros((1, 4, 3, 2))
    k = np.zeros((1, 3, 3, 2))
    with pytest.raises(ValueError):
        oracle.mha_fwd(q, k, k, scale=1.0)


# --------------------------------------------------------------------------
# the sublayer around the attention: projections with biases, head split,
# concatenation and the output projection
# --------------------------------------------------------------------------
def _sub_inputs(B, T, S, d, H, H_kv, seed=3):
    rng = np.random.default_rng(seed)
    dk = d // H
    x = rng.normal(size=(B, T, d))
    mem = rng.normal(size=(B, S, d))
    w_q = rng.normal(size=(d, H * dk)) / math.sqrt(d)
    w_k = rng.normal(size=(d, H_kv * dk)) / math.sqrt(d)
    w_v = rng.normal(size=(d, H_kv * dk)) / math.sqrt(d)
    w_o = rng.normal(size=(H * dk, d)) / math.sqrt(d)
    b = [rng.normal(size=n) * 0.1 for n in (H * dk, H_kv * dk, H_kv * dk, d)]
    return x, mem, w_q, w_k, w_v, w_o, b


def test_linear_brute_force():
    rng = np.random.default_rng(0)
    x, w, b = rng.normal(size=(2, 3, 4)), rng.normal(size=(4, 5)), rng.normal(size=5)
    y = oracle.linear(x, w, b)
    for i in range(2):
        for t in range(3):
            for o in range(5):
                acc = b[o]
                for c in range(4):
                    acc += x[i, t, c] * w[c, o]
                assert abs(y[i, t, o] - acc) < 1e-12


def test_linear_identity_adds_bias():
    x = np.random.default_rng(1).normal(size=(3, 6))
    b = np.arange(6.0)
    np.testing.assert_array_equal(oracle.linear(x, np.eye(6), b), x + b)
    np.testing.assert_array_equal(oracle.linear(x, np.eye(6)), x)


def test_linear_reads_bf16_bits_exactly():
    vals = np.array([[1.0, -2.5], [0.15625, 3.0]])
    bits = gen.f64_to_bf16_bits(vals)
    np.testing.assert_array_equal(oracle.linear(bits, gen.f64_to_bf16_bits(np.eye(2))),
                                  gen.bf16_bits_to_f64(bits))


@pytest.mark.parametrize("mask", [0, MASK_KEY_PADDING, MASK_CAUSAL])
def test_sublayer_zero_query_key_projections_average_values(oracle_lib, mask):
    # W_q = W_k = 0 and no q/k bias: every score is 0, each head averages the
    # value rows it may see, and the output is that average projected by W_o
    B, T, d, H = 2, 5, 8, 2
    S = T if mask & MASK_CAUSAL else 7
    x, mem, w_q, w_k, w_v, w_o, b = _sub_inputs(B, T, S, d, H, H)
    if mask & MASK_CAUSAL:
        mem = x
    lens = np.array([3, S], dtype=np.int32) if mask & MASK_KEY_PADDING else None
    out = oracle.mha_sublayer(x, mem, 0 * w_q, 0 * w_k, w_v, w_o, None, None, b[2], b[3], H=H,
                              mask_kind=mask, key_lengths=lens)
    v = mem @ w_v + b[2]
    for bi in range(B):
        for t in range(T):
            n = S
            if mask & MASK_KEY_PADDING:
                n = lens[bi]
            if mask & MASK_CAUSAL:
                n = t + 1
            mean = v[bi, :n].mean(axis=0)
            np.testing.assert_allclose(out[bi, t], mean @ w_o + b[3], rtol=0, atol=1e-12)


def test_sublayer_head_split_and_concat_order(oracle_lib):
    # with W_o = I and no output bias, output columns [i d_k, (i+1) d_k) are
    # head i: attention over the projections' columns [i d_k, (i+1) d_k)
    B, T, S, d, H = 2, 4, 6, 12, 3
    dk = d // H
    x, mem, w_q, w_k, w_v, _, b = _sub_inputs(B, T, S, d, H, H)
    out = oracle.mha_sublayer(x, mem, w_q, w_k, w_v, np.eye(d), b[0], b[1], b[2], None, H=H)
    for i in range(H):
        cols = slice(i * dk, (i + 1) * dk)
        q = (x @ w_q[:, cols] + b[0][cols])[:, None]
        k = (mem @ w_k[:, cols] + b[1][cols])[:, None]
        v = (mem @ w_v[:, cols] + b[2][cols])[:, None]
        head = oracle.mha_fwd(q, k, v, scale=1 / math.sqrt(dk))[:, 0]
        np.testing.assert_allclose(out[:, :, cols], head, rtol=0, atol=1e-12)


def test_sublayer_brute_force_tiny():
    # the whole sublayer from the definition with plain Python loops
    B, T, S, d, H = 1, 3, 4, 4, 2
    dk = d // H
    x, mem, w_q, w_k, w_v, w_o, b = _sub_inputs(B, T, S, d, H, H, seed=9)
    lens = np.array([3], dtype=np.int32)
    out = oracle.mha_sublayer(x, mem, w_q, w_k, w_v, w_o, *b, H=H, mask_kind=MASK_KEY_PADDING,
                              key_lengths=lens)

    def proj(rows, w, bias):
        return [[bias[o] + sum(r[c] * w[c][o] for c in range(len(r))) for o in range(len(bias))]
                for r in rows]
    q = proj(x[0].tolist(), w_q.tolist(), b[0].tolist())
    k = proj(mem[0].tolist(), w_k.tolist(), b[1].tolist())
    v = proj(mem[0].tolist(), w_v.tolist(), b[2].tolist())
    for t in range(T):
        concat = []
        for h in range(H):
            cs = range(h * dk, (h + 1) * dk)
            sc = [sum(q[t][c] * k[j][c] for c in cs) / math.sqrt(dk) for j in range(3)]
            e = [math.exp(z) for z in sc]
            wts = [z / sum(e) for z in e]
            concat += [sum(wts[j] * v[j][c] for j in range(3)) for c in cs]
        want = [b[3][o] + sum(concat[c] * w_o[c][o] for c in range(d)) for o in range(d)]
        np.testing.assert_allclose(out[0, t], want, rtol=0, atol=1e-12)


def test_sublayer_grouped_heads_equal_repeated_projections(oracle_lib):
    # sharing key/value heads equals giving every query head its own copy of
    # its group's key/value projection columns
    B, T, S, d, H, H_kv = 2, 5, 6, 16, 4, 2
    dk = d // H
    x, mem, w_q, w_k, w_v, w_o, b = _sub_inputs(B, T, S, d, H, H_kv)
    out = oracle.mha_sublayer(x, mem, w_q, w_k, w_v, w_o, *b, H=H, H_kv=H_kv)
    rep = lambda w: np.concatenate([w[..., (h // 2) * dk:(h // 2 + 1) * dk] for h in range(H)],
                                   axis=-1)
    out2 = oracle.mha_sublayer(x, mem, w_q, rep(w_k), rep(w_v), w_o, b[0], rep(b[1]), rep(b[2]),
                               b[3], H=H)
    np.testing.assert_allclose(out, out2, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# generation with a key/value cache: the queries are the last Lq positions
# --------------------------------------------------------------------------
from oracle import MASK_CAUSAL_TAIL  # noqa: E402


@pytest.mark.parametrize("Lq", [1, 3, 7])
def test_cached_decoding_equals_full_causal_rows(oracle_lib, Lq):
    # attending from the last Lq positions of a length-L sequence whose keys
    # and values are all cached gives exactly the last Lq rows of full causal
    # self-attention over the L positions
    B, H, L, d = 2, 3, 20, 8
    q, k, v = _rand(B, H, L, L, d, d, seed=11)
    full = oracle.mha_fwd(q, k, v, mask_kind=MASK_CAUSAL, scale=0.4)
    tail = oracle.mha_fwd(q[:, :, L - Lq:], k, v, mask_kind=MASK_CAUSAL_TAIL, scale=0.4)
    np.testing.assert_allclose(tail, full[:, :, L - Lq:], rtol=0, atol=1e-14)


def test_cached_decoding_with_lengths(oracle_lib):
    # per-sequence cache lengths: sequence b's queries sit at positions
    # len_b - Lq .. len_b - 1 and equal causal attention over its first len_b
    # positions; a cache shorter than Lq leaves the early queries without keys
    B, H, Lk, Lq, d = 3, 2, 16, 4, 8
    q, k, v = _rand(B, H, Lq, Lk, d, d, seed=12)
    lens = np.array([16, 9, 2], dtype=np.int32)
    out = oracle.mha_fwd(q, k, v, mask_kind=MASK_CAUSAL_TAIL | MASK_KEY_PADDING,
                         key_lengths=lens, scale=0.5)
    for b, lb in enumerate(lens):
        for i in range(Lq):
            pos = lb - Lq + i
            if pos < 0:
                assert np.all(out[b, :, i] == 0)
                continue
            one = oracle.mha_fwd(q[b:b + 1, :, i:i + 1], k[b:b + 1, :, :pos + 1],
                                 v[b:b + 1, :, :pos + 1], scale=0.5)
            np.testing.assert_allclose(out[b, :, i], one[0, :, 0], rtol=0, atol=1e-14)


def test_cached_decoding_single_query_is_key_padding(oracle_lib):
    B, H, Lk, d = 3, 2, 16, 8
    q, k, v = _rand(B, H, 1, Lk, d, d, seed=13)
    lens = np.array([16, 5, 1], dtype=np.int32)
    a = oracle.mha_fwd(q, k, v, mask_kind=MASK_CAUSAL_TAIL | MASK_KEY_PADDING, key_lengths=lens,
                       scale=0.3)
    b = oracle.mha_fwd(q, k, v, mask_kind=MASK_KEY_PADDING, key_lengths=lens, scale=0.3)
    np.testing.assert_array_equal(a, b)


def test_cached_decoding_rejects_mixed_causal(oracle_lib):
    q, k, v = _rand(1, 1, 4, 4, 4, 4)
    for m in (MASK_CAUSAL_TAIL | MASK_CAUSAL, MASK_CAUSAL_TAIL | MASK_QUERY_PADDING):
        with pytest.raises(ValueError):
            oracle.mha_fwd(q, k, v, mask_kind=m, key_lengths=np.array([4], np.int32), scale=1.0)
