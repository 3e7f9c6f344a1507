"""GPU parity for shared key/value heads (grouped- and multi-query attention)
and the [B, L, H, d] layout, through mha_fwd_ex, on all three kernels.

Same tolerances as the plain parity tests: fp32 max |err| <= 1e-4; bf16
max |err| <= 2e-2 and mean |err| <= 2e-3; padded and empty rows +0.0.
"""
import numpy as np
import pytest

import gen
import oracle
from helpers import check_case, run_gpu, spec

pytestmark = pytest.mark.gpu

C, KP, QP = gen.MASK_CAUSAL, gen.MASK_KEY_PADDING, gen.MASK_QUERY_PADDING


def _id(s):
    return "B%dH%dKV%dLq%dLk%dd%d_%s_m%d_%s" % (s["B"], s["H"], s["Hkv"], s["Lq"], s["Lk"],
                                                s["dk"], s["dtype"], s["mask"], s["layout"])


# shapes of the three workload families (short packed, causal decoder, cross)
# with every grouping of 8 query heads, in both layouts
FAMILIES = [
    dict(Lq=64, Lk=64, d=64, mask=KP | QP, len_range=(0, 64)),    # padded encoder
    dict(Lq=128, Lk=128, d=64, mask=C),                           # decoder
    dict(Lq=96, Lk=128, d=64, mask=KP, len_range=(16, 128)),      # cross, padded source
    dict(Lq=16, Lk=16, d=64, mask=C),                             # 8 heads in one tile
    dict(Lq=300, Lk=300, d=128, mask=C, amp=0.5),                 # long kernel
    dict(Lq=200, Lk=333, d=64, mask=KP, len_range=(0, 333)),      # long kernel, cross
]
GQA = [spec(3, 8, f["Lq"], f["Lk"], f["d"], mask=f["mask"], len_range=f.get("len_range"),
            amp=f.get("amp", 1.0), Hkv=hkv, layout=lay)
       for f in FAMILIES for hkv in (8, 4, 2, 1) for lay in ("bhsd", "bshd")]


@pytest.mark.parametrize("s", GQA, ids=_id)
def test_grouped_heads_and_layouts(s):
    check_case(s, seed=11)


# head counts that do not fill the last tile of packed pairs, and the fp32 path
ODD = [
    spec(2, 6, 32, 32, 64, mask=KP | QP, len_range=(0, 32), Hkv=2),      # P=4: 2 units/batch
    spec(2, 6, 32, 32, 64, mask=KP | QP, len_range=(0, 32), Hkv=3, layout="bshd"),
    spec(3, 5, 32, 32, 64, mask=C, Hkv=5, layout="bshd"),
    spec(3, 3, 16, 16, 64, mask=0, Hkv=1),                               # P capped at H
    spec(2, 12, 40, 40, 64, mask=KP, len_range=(1, 40), Hkv=4, layout="bshd"),
    spec(2, 4, 33, 33, 64, "f32", mask=KP | QP, len_range=(0, 33), Hkv=2),
    spec(2, 4, 45, 77, 100, "f32", mask=KP, len_range=(0, 77), Hkv=1, layout="bshd"),
    spec(2, 6, 50, 50, 17, "f32", mask=C, Hkv=3, layout="bshd"),
    spec(1, 4, 129, 129, 64, mask=C, Hkv=2, layout="bshd"),
    spec(1, 4, 513, 700, 128, mask=0, Hkv=1, layout="bshd"),
]


@pytest.mark.parametrize("s", ODD, ids=_id)
def test_partial_tiles_and_f32(s):
    check_case(s, seed=12)


def test_grouped_equals_repeated_heads_on_gpu():
    # sharing key/value head g among its group gives the same bits as giving
    # each query head its own copy of head g (plain multi-head attention)
    s = spec(2, 8, 128, 128, 64, mask=C, Hkv=2)
    q, k, v, _ = gen.make_inputs(s, seed=13)
    shared = run_gpu(q, k, v, None, s)
    s_rep = dict(s, Hkv=8)
    rep = run_gpu(q, np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1), None, s_rep)
    np.testing.assert_array_equal(shared, rep)


@pytest.mark.parametrize("L,d,mask", [(64, 64, KP | QP), (128, 64, C), (700, 128, C)])
def test_bshd_equals_transposed_bhsd_on_gpu(L, d, mask):
    # the same numbers in the other layout give the same bits, transposed
    s = spec(2, 4, L, L, d, mask=mask, len_range=(1, L) if mask & KP else None, Hkv=2)
    q, k, v, lens = gen.make_inputs(s, seed=14)
    a = run_gpu(q, k, v, lens, s)
    t = lambda x: np.ascontiguousarray(x.transpose(0, 2, 1, 3))
    b = run_gpu(t(q), t(k), t(v), lens, dict(s, layout="bshd"))
    np.testing.assert_array_equal(t(b), a)


def test_long_gqa_sampled_rows():
    # long causal shape with 16 query heads over 4 key/value heads
    s = spec(1, 16, 4096, 4096, 128, mask=C, amp=0.5, Hkv=4, layout="bshd")
    L = s["Lq"]
    rng = np.random.default_rng(2)
    picks = []
    for bh in range(16):
        picks += [bh * L + i for i in (0, 127, 128, 2047, L - 129, L - 1)]
        picks += list(bh * L + rng.integers(0, L, 8))
    check_case(s, seed=15, rows=np.array(sorted(set(picks)), dtype=np.int64))


def test_ex_rejects_bad_groups():
    import torch
    import transformer_head_scaled_mha_gb300 as mha
    q = torch.zeros(1, 6, 16, 64, device="cuda", dtype=torch.bfloat16)
    k = torch.zeros(1, 4, 16, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(mha.MhaError):
        mha.mha_fwd_ex(q, k, k)
    with pytest.raises(ValueError):
        mha.mha_fwd(q, k, k)  # the plain entry point needs H_kv == H
