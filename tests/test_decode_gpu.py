"""GPU parity for generation with a key/value cache (MHA_MASK_CAUSAL_TAIL):
the Lq queries are the last Lq positions of each sequence, whose len_b keys
and values are in the cache.  All three kernels, both layouts, shared
key/value heads.  Tolerances as in test_parity_gpu.py."""
import numpy as np
import pytest

import gen
import oracle
from helpers import check_case, compare, run_gpu, spec

pytestmark = pytest.mark.gpu

KP, TAIL, C = gen.MASK_KEY_PADDING, gen.MASK_CAUSAL_TAIL, gen.MASK_CAUSAL


def _id(s):
    return "B%dH%dKV%dLq%dLk%dd%d_%s_m%d_%s" % (s["B"], s["H"], s["Hkv"], s["Lq"], s["Lk"],
                                                s["dk"], s["dtype"], s["mask"], s["layout"])


CASES = [
    # one new token against caches of various lengths (typical decoding step)
    spec(8, 8, 1, 100, 64, mask=TAIL | KP, len_range=(1, 100)),
    spec(4, 32, 1, 128, 64, mask=TAIL | KP, len_range=(1, 128), Hkv=8, layout="bshd"),
    spec(4, 16, 1, 1000, 128, mask=TAIL | KP, len_range=(1, 1000), Hkv=4, layout="bshd"),
    spec(2, 8, 1, 8192, 128, mask=TAIL | KP, len_range=(4000, 8192), amp=0.5, Hkv=1,
         layout="bshd"),
    spec(3, 4, 1, 300, 64, mask=TAIL),
    # a few tokens at once (speculative or chunked steps)
    spec(4, 8, 4, 128, 64, mask=TAIL | KP, len_range=(0, 128)),
    spec(4, 8, 16, 128, 64, mask=TAIL | KP, len_range=(8, 128), Hkv=2, layout="bshd"),
    spec(2, 8, 33, 100, 64, mask=TAIL),
    spec(2, 4, 300, 1000, 128, mask=TAIL | KP, len_range=(200, 1000)),
    spec(2, 4, 129, 777, 64, mask=TAIL, layout="bshd"),
    # fp32 path
    spec(2, 4, 3, 90, 64, "f32", mask=TAIL | KP, len_range=(0, 90)),
    spec(2, 4, 40, 70, 100, "f32", mask=TAIL, Hkv=2, layout="bshd"),
]


@pytest.mark.parametrize("s", CASES, ids=_id)
def test_cached_decoding_parity(s):
    check_case(s, seed=21)


@pytest.mark.parametrize("L,d,dt", [(128, 64, "bf16"), (300, 128, "bf16"), (40, 64, "f32")])
def test_tail_over_whole_sequence_is_causal(L, d, dt):
    # Lq = Lk = len: the cached-decoding mask is the causal mask
    s = spec(2, 4, L, L, d, dt, mask=TAIL)
    q, k, v, _ = gen.make_inputs(s, seed=5)
    a = run_gpu(q, k, v, None, s)
    b = run_gpu(q, k, v, None, dict(s, mask=C))
    ref = oracle.mha_fwd(q, k, v, mask_kind=C, scale=gen.default_scale(d))
    compare(a, ref, dt)
    compare(b, ref, dt)


def test_queries_before_the_cache_are_zero():
    # len_b < Lq: the first Lq - len_b queries have no key at all -> +0.0
    s = spec(3, 4, 8, 64, 64, mask=TAIL | KP)
    q, k, v, _ = gen.make_inputs(s, seed=6)
    lens = np.array([3, 0, 64], dtype=np.int32)
    out = run_gpu(q, k, v, lens, s)
    ref = oracle.mha_fwd(q, k, v, mask_kind=TAIL | KP, key_lengths=lens,
                         scale=gen.default_scale(64))
    compare(out, ref, "bf16")
    assert np.all(out[0, :, :5] == 0) and np.all(out[1] == 0)


def test_cached_step_equals_rows_of_full_causal():
    # the last Lq rows of causal attention over L positions, computed as a
    # decoding step over the cache of all L keys and values
    L, Lq = 200, 5
    s = spec(2, 4, L, L, 128, mask=C)
    q, k, v, _ = gen.make_inputs(s, seed=7)
    full = run_gpu(q, k, v, None, s)
    step = run_gpu(np.ascontiguousarray(q[:, :, L - Lq:]), k, v, None,
                   spec(2, 4, Lq, L, 128, mask=TAIL))
    ref = oracle.mha_fwd(q, k, v, mask_kind=C, scale=gen.default_scale(128))[:, :, L - Lq:]
    compare(step, ref, "bf16")
    compare(full[:, :, L - Lq:], ref, "bf16")
