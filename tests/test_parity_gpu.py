"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Tolerances (written here, from the target): fp32 max |err| <= 1e-4; bf16
max |err| <= 2e-2 and mean |err| <= 2e-3; padded query rows and rows with no
allowed key are +0.0 bit for bit.
"""
import numpy as np
import pytest

import gen
import oracle
from helpers import check_case, compare, run_gpu, spec

pytestmark = pytest.mark.gpu

C, KP, QP = gen.MASK_CAUSAL, gen.MASK_KEY_PADDING, gen.MASK_QUERY_PADDING


# ---------------------------------------------------------------------------
# the five workloads at their full sizes (rows sampled where the oracle is slow)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["enc_f32_b2_h8_l32_d64", "enc_pad_bf16_b256_h8_l64_d64",
                                  "dec_causal_bf16_b128_h8_l128_d64",
                                  "cross_pad_bf16_b64_h16_lq96_lk128_d64"])
def test_workload_full_size_all_rows(name):
    check_case(gen.WORKLOADS[name], label=name)


def test_long_causal_full_size_sampled_rows():
    s = gen.WORKLOADS["long_causal_bf16_b4_h16_l8192_d128"]
    B, H, L = s["B"], s["H"], s["Lq"]
    rng = np.random.default_rng(1)
    picks = []
    for bh in range(B * H):
        # first rows, tile edges, last rows, and random rows of every head
        fixed = [0, 1, 127, 128, 255, 256, 4095, 4096, L - 129, L - 128, L - 2, L - 1]
        picks += [bh * L + i for i in fixed]
        picks += list(bh * L + rng.integers(0, L, 20))
    rows = np.array(sorted(set(picks)), dtype=np.int64)
    check_case(s, rows=rows, label="long_causal full (sampled)")


# ---------------------------------------------------------------------------
# scaled-down workloads: every row, several tiles and ragged tails
# ---------------------------------------------------------------------------
SMALL = [
    spec(2, 3, 33, 33, 64, "f32"),
    spec(2, 3, 45, 77, 100, "f32", mask=KP, len_range=(0, 77)),
    spec(3, 2, 50, 50, 17, "f32", mask=C),
    spec(3, 2, 40, 40, 128, "f32", mask=KP | QP, len_range=(0, 40)),
    spec(8, 4, 64, 64, 64, mask=KP | QP, len_range=(0, 64)),
    spec(5, 3, 128, 128, 64, mask=C),
    spec(6, 3, 96, 128, 64, mask=KP, len_range=(0, 128)),
    spec(3, 5, 7, 13, 64, mask=KP, len_range=(1, 13)),
    spec(4, 4, 1, 1, 64),
    spec(4, 3, 16, 16, 64, mask=C),
    spec(5, 3, 30, 20, 64, mask=KP, len_range=(0, 20)),
    spec(7, 3, 40, 40, 64, mask=KP | QP, len_range=(0, 40)),
    spec(2, 2, 100, 100, 64, mask=C | KP, len_range=(0, 100)),
    spec(3, 3, 30, 30, 64, mask=0),
    spec(1, 2, 700, 700, 128, mask=C, amp=0.5),
    spec(1, 2, 513, 513, 128, mask=0),
    spec(2, 2, 300, 1000, 128, mask=KP, len_range=(0, 1000)),
    spec(2, 2, 257, 257, 64, mask=C),
    spec(2, 2, 129, 200, 64),
    spec(2, 1, 400, 400, 128, mask=KP | QP, len_range=(0, 400)),
    spec(2, 2, 130, 130, 128, mask=C | KP, len_range=(100, 130)),
]


@pytest.mark.parametrize("s", SMALL, ids=lambda s: "B%dH%dLq%dLk%dd%d_%s_m%d" % (
    s["B"], s["H"], s["Lq"], s["Lk"], s["dk"], s["dtype"], s["mask"]))
def test_small_all_rows(s):
    check_case(s, seed=5)


@pytest.mark.parametrize("L", [1, 7, 63, 65, 127, 129, 255, 1023])
@pytest.mark.parametrize("d", [64, 128])
def test_odd_lengths_causal(L, d):
    check_case(spec(1, 2, L, L, d, mask=C), seed=L)


@pytest.mark.parametrize("d", [64, 128])
def test_odd_lengths_long_tail_8191(d):
    s = spec(1, 1, 8191, 8191, d, mask=C)
    rows = np.array([0, 1, 4000, 8063, 8064, 8189, 8190], dtype=np.int64)
    check_case(s, seed=3, rows=rows)


# ---------------------------------------------------------------------------
# masking properties on the GPU
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("L,d", [(128, 64), (300, 128)])
def test_future_tokens_never_change_earlier_rows(L, d):
    s = spec(1, 2, L, L, d, mask=C)
    q, k, v, _ = gen.make_inputs(s, seed=9)
    base = run_gpu(q, k, v, None, s)
    for t in (0, 1, L // 2, L - 1):
        k2, v2 = k.copy(), v.copy()
        k2[:, :, t:] = gen.f64_to_bf16_bits(np.full(k2[:, :, t:].shape, 3.0))
        v2[:, :, t:] = gen.f64_to_bf16_bits(np.full(v2[:, :, t:].shape, -5.0))
        out = run_gpu(q, k2, v2, None, s)
        np.testing.assert_array_equal(out[:, :, :t], base[:, :, :t])


@pytest.mark.parametrize("Lq,Lk,d,mask", [(64, 64, 64, KP | QP), (96, 128, 64, KP),
                                          (200, 400, 128, KP)])
def test_padded_keys_never_matter(Lq, Lk, d, mask):
    s = spec(4, 2, Lq, Lk, d, mask=mask, len_range=(1, Lk))
    q, k, v, lens = gen.make_inputs(s, seed=4)
    base = run_gpu(q, k, v, lens, s)
    k2, v2 = k.copy(), v.copy()
    for b, lb in enumerate(lens):
        k2[b, :, lb:] = gen.f64_to_bf16_bits(np.full(k2[b, :, lb:].shape, 50.0))
        v2[b, :, lb:] = gen.f64_to_bf16_bits(np.full(v2[b, :, lb:].shape, -70.0))
    out = run_gpu(q, k2, v2, lens, s)
    np.testing.assert_array_equal(out, base)


@pytest.mark.parametrize("Lq,Lk,d", [(64, 64, 64), (300, 300, 128), (33, 33, 64)])
def test_degenerate_lengths(Lq, Lk, d):
    # lengths 0 (no key at all: +0 rows), 1 (output = V[0]), Lk, and out of
    # range values (clamped)
    for dt in ("bf16", "f32"):
        s = spec(5, 2, Lq, Lk, d, dtype=dt, mask=KP | QP)
        q, k, v, _ = gen.make_inputs(s, seed=2)
        lens = np.array([0, 1, Lk, -3, Lk + 10], dtype=np.int32)
        out = run_gpu(q, k, v, lens, s)
        ref = oracle.mha_fwd(q, k, v, mask_kind=KP | QP, key_lengths=lens,
                             scale=gen.default_scale(d))
        compare(out, ref, dt)
        assert np.all(out[0] == 0) and np.all(out[3] == 0)


def test_no_keys_writes_zeros():
    import torch
    import transformer_head_scaled_mha_gb300 as mha
    for dt in (torch.float32, torch.bfloat16):
        q = torch.randn(2, 2, 5, 64, device="cuda").to(dt)
        k = torch.empty(2, 2, 0, 64, device="cuda", dtype=dt)
        out = torch.full((2, 2, 5, 64), 7.0, device="cuda", dtype=dt)
        mha.mha_fwd(q, k, k, out)
        torch.cuda.synchronize()
        assert torch.all(out == 0) and not torch.any(torch.signbit(out))


def test_empty_problem_is_noop():
    import torch
    import transformer_head_scaled_mha_gb300 as mha
    q = torch.empty(0, 2, 5, 64, device="cuda", dtype=torch.bfloat16)
    out = mha.mha_fwd(q, q, q)
    assert out.shape == (0, 2, 5, 64)


@pytest.mark.parametrize("Lq,Lk,d,mask", [(128, 128, 64, C), (64, 64, 64, 0), (96, 128, 64, KP),
                                          (16, 16, 64, C), (300, 300, 128, C),
                                          (200, 333, 64, KP)])
def test_scores_climbing_along_keys(Lq, Lk, d, mask):
    # scores that rise by about 10 (log2 units) every 32 keys: each later key
    # block's max far exceeds the earlier ones, which is where a kernel that
    # takes exponents against a provisional max must correct what it wrote
    rng = np.random.default_rng(7)
    B, H = 2, 2
    q = np.abs(rng.normal(size=(B, H, Lq, d))) * 0.5 + 0.5
    ramp = (np.arange(Lk) / 16.0)[None, None, :, None] * (64.0 / d)
    k = ramp * (0.5 + 0.1 * rng.normal(size=(B, H, Lk, d)))
    v = rng.normal(size=(B, H, Lk, d))
    q, k, v = (gen.f64_to_bf16_bits(x) for x in (q, k, v))
    lens = np.array([Lk - 5, min(Lk, 70)], dtype=np.int32) if mask & KP else None
    s = spec(B, H, Lq, Lk, d, mask=mask)
    out = run_gpu(q, k, v, lens, s)
    ref = oracle.mha_fwd(q, k, v, mask_kind=mask, key_lengths=lens, scale=gen.default_scale(d))
    compare(out, ref, "bf16", label="climbing scores")
    # and the reverse: the first key block holds the largest scores
    k2 = np.ascontiguousarray(k[:, :, ::-1])
    out = run_gpu(q, k2, v, lens, s)
    ref = oracle.mha_fwd(q, k2, v, mask_kind=mask, key_lengths=lens, scale=gen.default_scale(d))
    compare(out, ref, "bf16", label="falling scores")


@pytest.mark.parametrize("scale", [0.0, 1.0, -0.3])
def test_other_scales(scale):
    check_case(spec(2, 2, 96, 128, 64), scale=scale, seed=8)
    check_case(spec(1, 2, 300, 300, 128, mask=C), scale=scale, seed=8)
    check_case(spec(2, 2, 40, 40, 64, "f32", mask=C), scale=scale, seed=8)
    # masked rows on the packed kernel (a zero scale must not meet a masked -inf)
    check_case(spec(2, 2, 128, 128, 64, mask=C), scale=scale, seed=8)
    check_case(spec(3, 2, 64, 64, 64, mask=KP | QP, len_range=(0, 64)), scale=scale, seed=8)


def test_deterministic():
    s = gen.WORKLOADS["enc_pad_bf16_b256_h8_l64_d64"]
    q, k, v, lens = gen.make_inputs(s, seed=0)
    a = run_gpu(q, k, v, lens, s)
    b = run_gpu(q, k, v, lens, s)
    np.testing.assert_array_equal(a, b)
    s2 = spec(1, 4, 1000, 1000, 128, mask=C)
    q, k, v, _ = gen.make_inputs(s2, seed=0)
    np.testing.assert_array_equal(run_gpu(q, k, v, None, s2), run_gpu(q, k, v, None, s2))


def test_worked_example_on_gpu():
    # the pages' three-token example (identity projections), padded to d = 64
    # with zero columns, which changes no dot product; fp32 path
    import json, math, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")))
    for name, c in g["cases"].items():
        X = np.zeros((1, 1, 3, 64), dtype=np.float32)
        X[0, 0, :, :2] = np.array(c["X"], dtype=np.float32)
        scale = 1 / math.sqrt(2) if c["scale"] == "1/sqrt(2)" else 1.0
        s = spec(1, 1, 3, 3, 64, "f32")
        out = run_gpu(X, X, X, None, s, scale=scale)
        for row, vals in c["out"].items():
            np.testing.assert_allclose(out[0, 0, int(row), :2], vals, atol=1e-5)


def test_debug_status_clean():
    import transformer_head_scaled_mha_gb300 as mha
    check_case(spec(2, 2, 64, 64, 64, mask=KP | QP, len_range=(0, 64)))
    assert mha.mha_debug_status() == mha.MHA_OK
