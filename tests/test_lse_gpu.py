"""GPU parity of the row statistics that mha_fwd_lse writes beside the output.

For query row i of head (b, h) the statistic is the base-2 log of the softmax
denominator over the allowed keys A_i (the scaled dot-product attention of
"Attention Is All You Need", section 3.2.1, with the masks of section 3.2.3):

  lse_i = log2( sum_{j in A_i} exp(s_ij) ),   s_ij = scale * q_i . k_j

and +inf for a row that is stored as zeros (A_i empty, or a padded query).
The oracle's scaled logits s_ij give it directly (a numpy logsumexp over the
row, divided by ln 2).  Error bounds: fp32 paths 1e-4 + 1e-5 |lse|; bf16 paths
4e-3 + 1e-5 |lse| (the denominator is summed in fp32 from weights that may be
rounded to bf16 first: relative 2^-9 at most, 2^-9 / ln 2 in log2).
"""
import numpy as np
import pytest

import gen
import oracle
from helpers import from_device, spec, to_device

pytestmark = pytest.mark.gpu

C, KP, QP, TAIL = gen.MASK_CAUSAL, gen.MASK_KEY_PADDING, gen.MASK_QUERY_PADDING, \
    gen.MASK_CAUSAL_TAIL
LSE_TOL = {"f32": (1e-4, 1e-5), "bf16": (4e-3, 1e-5)}


def lse_from_scores(sc):
    """log2 of sum_j exp(s_j) along the last axis; +inf where every s_j is -inf."""
    m = sc.max(axis=-1, keepdims=True)
    dead = ~np.isfinite(m[..., 0])
    mm = np.where(np.isfinite(m), m, 0.0)
    with np.errstate(under="ignore", divide="ignore"):
        r = (mm[..., 0] + np.log(np.exp(sc - mm).sum(axis=-1))) / np.log(2.0)
    r[dead] = np.inf
    return r


def check_lse(got, ref, dtype, label):
    inf_ref = np.isposinf(ref)
    assert np.array_equal(np.isposinf(got), inf_ref), "%s: +inf rows differ" % label
    assert np.isfinite(got[~inf_ref]).all(), "%s: non-finite statistic" % label
    a, r = LSE_TOL[dtype]
    err = np.abs(got[~inf_ref] - ref[~inf_ref])
    bound = a + r * np.abs(ref[~inf_ref])
    assert np.all(err <= bound), "%s: max err %.3g" % (label, float(err.max()))


def _id(s):
    return "B%dH%dKV%dLq%dLk%dd%d_%s_m%d_%s" % (s["B"], s["H"], s["Hkv"], s["Lq"], s["Lk"],
                                                s["dk"], s["dtype"], s["mask"], s["layout"])


CASES = [
    # fp32 path
    spec(2, 3, 45, 77, 100, "f32", mask=KP, len_range=(0, 77)),
    spec(2, 2, 40, 40, 128, "f32", mask=KP | QP, len_range=(0, 40), layout="bshd"),
    # packed short path (d 64, at most 128 rows and keys)
    spec(4, 2, 64, 64, 64, mask=KP | QP, len_range=(0, 64)),
    spec(2, 4, 128, 128, 64, mask=C, Hkv=2),
    spec(3, 8, 20, 100, 64, mask=KP, len_range=(0, 100), layout="bshd"),
    # long path: several key tiles, ragged tails, both head sizes
    spec(1, 2, 300, 300, 128, mask=C, amp=0.5),
    spec(2, 2, 200, 333, 64, mask=KP, len_range=(0, 333)),
    spec(2, 4, 260, 700, 64, mask=TAIL | KP, len_range=(300, 700), Hkv=1, layout="bshd"),
    spec(1, 2, 513, 513, 128, mask=C | KP, len_range=(100, 513)),
    # decode path: one or two rows per key/value head
    spec(3, 2, 1, 500, 64, mask=TAIL | KP, len_range=(1, 500)),
    spec(2, 8, 2, 300, 128, mask=KP, len_range=(0, 300), Hkv=4),
]


@pytest.mark.parametrize("s", CASES, ids=_id)
def test_forward_lse_matches_oracle(s):
    import torch
    import transformer_head_scaled_mha_gb300 as mha
    q, k, v, lens = gen.make_inputs(s, seed=51)
    dt, layout = s["dtype"], s["layout"]
    scale = gen.default_scale(s["dk"])
    kl = torch.from_numpy(lens).cuda() if lens is not None else None
    Q, K, V = (to_device(a, dt) for a in (q, k, v))
    out, lse = mha.mha_fwd_lse(Q, K, V, layout=layout, mask_kind=s["mask"], key_lengths=kl,
                               scale=scale)
    ref_out = mha.mha_fwd_ex(Q, K, V, layout=layout, mask_kind=s["mask"], key_lengths=kl,
                             scale=scale)
    torch.cuda.synchronize()
    assert mha.mha_debug_status() == mha.MHA_OK
    assert np.array_equal(from_device(out), from_device(ref_out)), "output differs from mha_fwd_ex"
    _, sc = oracle.mha_fwd(q, k, v, mask_kind=s["mask"], key_lengths=lens, scale=scale,
                           return_scores=True, layout=layout)
    check_lse(lse.cpu().numpy().astype(np.float64), lse_from_scores(sc), dt, _id(s))


def test_forward_lse_no_keys_is_inf():
    import torch
    import transformer_head_scaled_mha_gb300 as mha
    q = torch.randn(2, 3, 5, 64, device="cuda").bfloat16()
    k = torch.empty(2, 3, 0, 64, device="cuda", dtype=torch.bfloat16)
    out, lse = mha.mha_fwd_lse(q, k, k)
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(torch.isposinf(lse))


def test_forward_lse_long_causal_full_size_sampled():
    # the long causal workload at full size: first and last rows of a few heads
    import torch
    import transformer_head_scaled_mha_gb300 as mha
    s = gen.WORKLOADS["long_causal_bf16_b4_h16_l8192_d128"]
    L, H = s["Lq"], s["H"]
    q, k, v, _ = gen.make_inputs(s, seed=52)
    scale = gen.default_scale(s["dk"])
    Q, K, V = (to_device(a, "bf16") for a in (q, k, v))
    _, lse = mha.mha_fwd_lse(Q, K, V, mask_kind=C, scale=scale)
    torch.cuda.synchronize()
    assert mha.mha_debug_status() == mha.MHA_OK
    got = lse.cpu().numpy().astype(np.float64).reshape(-1)
    del Q, K, V
    rows = []
    for u in (0, 21, 63):
        rows += [u * L + i for i in (0, 1, 127, 128, 4097, L - 2, L - 1)]
    _, sc = oracle.mha_fwd(q, k, v, mask_kind=C, scale=scale, rows=rows, return_scores=True)
    check_lse(got[rows], lse_from_scores(sc), "bf16", "long causal sampled")
