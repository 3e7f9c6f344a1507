"""GPU parity for the projection kernel (mha_linear_fwd) and the whole
multi-head sublayer (mha_sublayer_fwd) against the fp64 oracle.

Tolerances, from the arithmetic:
- linear: the exact product is rounded once to bf16 (relative 2^-9) after an
  fp32 accumulation; elementwise |err| <= 2^-8 |ref| + 2e-4.
- sublayer: q, k, v, P, the concatenated heads and the output are each
  rounded to bf16; emulating those roundings in fp64 on these workloads gives
  max |err| 0.006-0.010 and mean |err| 5-7e-4, so the bounds are max 3e-2 and
  mean 3e-3.  Rows whose attention is padding (query padding) reduce to the
  output bias exactly.
"""
import math

import numpy as np
import pytest

import gen
import oracle
from helpers import from_device, to_device

pytestmark = pytest.mark.gpu


def _bf(a):
    return gen.f64_to_bf16_bits(a)


def _f(a):
    return gen.bf16_bits_to_f64(a)


def _linear_case(M, K, N, seed, bias=True):
    rng = np.random.default_rng(seed)
    x = _bf(rng.normal(size=(M, K)))
    w = _bf(rng.normal(size=(K, N)) / math.sqrt(K))
    b = _bf(rng.normal(size=N) * 0.5) if bias else None
    return x, w, b


@pytest.mark.parametrize("M,K,N", [(1000, 512, 512), (128, 64, 64), (300, 256, 72),
                                   (5, 1024, 1536), (129, 200, 136), (1, 8, 8),
                                   (16384, 512, 512), (777, 192, 320), (2000, 448, 64),
                                   (3000, 512, 1536)])
def test_linear_parity(M, K, N):
    import transformer_head_scaled_mha_gb300 as mha
    x, w, b = _linear_case(M, K, N, seed=M + K + N)
    y = from_device(mha.mha_linear_fwd(to_device(x, "bf16"), to_device(w, "bf16"),
                                       to_device(b, "bf16")))
    ref = oracle.linear(x, w, b)
    err = np.abs(_f(y) - ref)
    assert np.all(err <= 2.0 ** -8 * np.abs(ref) + 2e-4), float(err.max())


def test_linear_without_bias_and_batched_input():
    import transformer_head_scaled_mha_gb300 as mha
    x, w, _ = _linear_case(3 * 70, 128, 192, seed=4, bias=False)
    x3 = x.reshape(3, 70, 128)
    y = from_device(mha.mha_linear_fwd(to_device(x3, "bf16"), to_device(w, "bf16")))
    ref = oracle.linear(x3, w)
    assert y.shape == (3, 70, 192)
    err = np.abs(_f(y) - ref)
    assert np.all(err <= 2.0 ** -8 * np.abs(ref) + 2e-4)


def test_linear_identity_is_exact():
    # W = I, b = 0: every output is one input times 1 plus zeros -> exact
    import transformer_head_scaled_mha_gb300 as mha
    x, _, _ = _linear_case(257, 136, 8, seed=5)
    w = _bf(np.eye(136))
    b = _bf(np.zeros(136))
    y = from_device(mha.mha_linear_fwd(to_device(x, "bf16"), to_device(w, "bf16"),
                                       to_device(b, "bf16")))
    np.testing.assert_array_equal(y, x)


def _sub_case(B, T, S, d, H, H_kv, mask, seed, cross):
    rng = np.random.default_rng(seed)
    dk = d // H
    x = _bf(rng.normal(size=(B, T, d)))
    mem = _bf(rng.normal(size=(B, S, d))) if cross else None
    w = [_bf(rng.normal(size=(d, n)) / math.sqrt(d)) for n in (H * dk, H_kv * dk, H_kv * dk)]
    w.append(_bf(rng.normal(size=(H * dk, d)) / math.sqrt(H * dk)))
    b = [_bf(rng.normal(size=n) * 0.1) for n in (H * dk, H_kv * dk, H_kv * dk, d)]
    lens = None
    if mask & (gen.MASK_KEY_PADDING | gen.MASK_QUERY_PADDING):
        lens = rng.integers(0, S + 1, size=B).astype(np.int32)
        lens[0] = S
    return x, mem, w, b, lens


SUB = [
    # B, T, S, d_model, H, H_kv, mask, cross
    (8, 64, 64, 512, 8, 8, gen.MASK_KEY_PADDING | gen.MASK_QUERY_PADDING, False),
    (4, 128, 128, 512, 8, 8, gen.MASK_CAUSAL, False),
    (4, 96, 128, 1024, 16, 16, gen.MASK_KEY_PADDING, True),
    (2, 64, 80, 512, 8, 2, gen.MASK_KEY_PADDING, True),
    (2, 50, 50, 1024, 8, 8, gen.MASK_CAUSAL | gen.MASK_KEY_PADDING, False),
    (1, 300, 300, 512, 8, 8, gen.MASK_CAUSAL, False),
    (2, 40, 300, 512, 8, 1, 0, True),
]


@pytest.mark.parametrize("case", SUB, ids=lambda c: "B%dT%dS%dd%dH%dKV%d_m%d_%s" % (
    c[0], c[1], c[2], c[3], c[4], c[5], c[6], "cross" if c[7] else "self"))
def test_sublayer_parity(case):
    import torch
    import transformer_head_scaled_mha_gb300 as mha
    B, T, S, d, H, H_kv, mask, cross = case
    x, mem, w, b, lens = _sub_case(B, T, S, d, H, H_kv, mask, seed=B * T + S, cross=cross)
    kl = torch.from_numpy(lens).cuda() if lens is not None else None
    dev = lambda a: to_device(a, "bf16") if a is not None else None
    out = mha.mha_sublayer_fwd(dev(x), *[dev(t) for t in w], *[dev(t) for t in b],
                               mem=dev(mem), H=H, H_kv=H_kv, mask_kind=mask, key_lengths=kl)
    torch.cuda.synchronize()
    got = _f(from_device(out))
    ref = oracle.mha_sublayer(x, mem if cross else x, *w, *b, H=H, H_kv=H_kv, mask_kind=mask,
                              key_lengths=lens)
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    assert err.max() <= 3e-2 and err.mean() <= 3e-3, (float(err.max()), float(err.mean()))
    if mask & gen.MASK_QUERY_PADDING:
        # padded query rows: no attention, the output is the bias
        for bi, lb in enumerate(lens):
            np.testing.assert_array_equal(from_device(out)[bi, lb:],
                                          np.broadcast_to(b[3], (T - lb, d)))
    assert mha.mha_debug_status() == mha.MHA_OK


def test_sublayer_with_caller_workspace_twice():
    # the same call twice with one caller-owned workspace gives the same bits
    import torch
    import transformer_head_scaled_mha_gb300 as mha
    B, T, d, H = 4, 64, 512, 8
    x, _, w, b, lens = _sub_case(B, T, T, d, H, H, gen.MASK_KEY_PADDING, seed=3, cross=False)
    n = mha.mha_sublayer_workspace_size(B, T, T, d, H, H, 64, 64)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    kl = torch.from_numpy(lens).cuda()
    dev = lambda a: to_device(a, "bf16")
    args = (dev(x), *[dev(t) for t in w], *[dev(t) for t in b])
    o1 = from_device(mha.mha_sublayer_fwd(*args, H=H, mask_kind=gen.MASK_KEY_PADDING,
                                          key_lengths=kl, workspace=ws))
    o2 = from_device(mha.mha_sublayer_fwd(*args, H=H, mask_kind=gen.MASK_KEY_PADDING,
                                          key_lengths=kl, workspace=ws))
    np.testing.assert_array_equal(o1, o2)


def test_sublayer_without_keys_gives_bias():
    # S = 0: every query attends to nothing (+0 heads), so out = b_o exactly
    import torch
    import transformer_head_scaled_mha_gb300 as mha
    x, _, w, b, _ = _sub_case(2, 16, 16, 512, 8, 8, 0, seed=1, cross=False)
    mem = torch.empty(2, 0, 512, dtype=torch.bfloat16, device="cuda")
    dev = lambda a: to_device(a, "bf16")
    out = mha.mha_sublayer_fwd(dev(x), *[dev(t) for t in w], *[dev(t) for t in b], mem=mem, H=8)
    np.testing.assert_array_equal(from_device(out), np.broadcast_to(b[3], (2, 16, 512)))
