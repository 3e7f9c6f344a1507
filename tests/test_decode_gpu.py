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


# ---------------------------------------------------------------------------
# the few-query kernel: keys on the tensor-memory lanes, at most 16 query rows
# ((H / H_kv) * Lq) per key/value head; masks NONE, KEY_PADDING, CAUSAL_TAIL
# ---------------------------------------------------------------------------
DECODE_PATH = 5


def _path(s):
    import transformer_head_scaled_mha_gb300 as mha
    return mha.mha_fwd_path_ex(s["B"], s["H"], s.get("Hkv", s["H"]), s["Lq"], s["Lk"], s["dk"], s["dv"],
                               s["mask"], 1 if s["dtype"] == "bf16" else 0)


FEW = [
    spec(5, 8, 1, 1000, 64, mask=TAIL | KP, len_range=(0, 1000), layout="bshd"),
    spec(3, 8, 1, 777, 128, mask=TAIL | KP, len_range=(1, 777), Hkv=2, layout="bshd"),
    spec(2, 16, 1, 2049, 64, mask=TAIL, Hkv=1),                            # 16 rows
    spec(4, 4, 4, 513, 64, mask=TAIL | KP, len_range=(0, 513)),
    spec(3, 8, 8, 300, 128, mask=TAIL, Hkv=4, layout="bshd"),              # 16 rows
    spec(2, 4, 4, 1111, 128, mask=KP, len_range=(100, 1111), Hkv=1, layout="bshd"),
    spec(3, 6, 5, 400, 64, mask=0, Hkv=3),                                 # 10 rows
    spec(2, 2, 16, 256, 64, mask=TAIL),                                    # 2 whole tiles
    spec(2, 2, 3, 100, 128, mask=TAIL | KP, len_range=(0, 100)),           # one ragged tile
    spec(1, 1, 1, 129, 64),
    spec(2, 4, 2, 4096, 128, mask=TAIL | KP, len_range=(1000, 4096), amp=0.5, Hkv=1),
    # more pairs than CTAs: each CTA walks many pairs, some of them empty
    spec(160, 8, 1, 300, 64, mask=TAIL | KP, len_range=(0, 300), layout="bshd"),
    spec(40, 16, 2, 500, 128, mask=TAIL | KP, len_range=(0, 500), Hkv=8, layout="bshd"),
]


@pytest.mark.parametrize("s", FEW, ids=_id)
def test_few_query_kernel_parity(s):
    assert _path(s) == DECODE_PATH
    check_case(s, seed=31)


@pytest.mark.parametrize("d", [64, 128])
def test_few_query_kernel_length_edges(d):
    # cache lengths at and around tile edges, and empty caches between full ones
    s = spec(12, 4, 2, 700, d, mask=TAIL | KP, Hkv=2, layout="bshd")
    assert _path(s) == DECODE_PATH
    q, k, v, _ = gen.make_inputs(s, seed=32)
    lens = np.array([0, 1, 127, 128, 129, 255, 256, 257, 0, 699, 700, 0], dtype=np.int32)
    out = run_gpu(q, k, v, lens, s)
    ref = oracle.mha_fwd(q, k, v, mask_kind=TAIL | KP, key_lengths=lens,
                         scale=gen.default_scale(d), layout="bshd")
    compare(out, ref, "bf16", label="length edges")
    assert np.all(out[lens == 0] == 0)
    # one key: the output row is that key's value row, rounded once
    np.testing.assert_array_equal(out[1, 1], v[1, 0, [0, 0, 1, 1]])
    # and every cache empty: all +0.0
    zero = run_gpu(q, k, v, np.zeros(12, dtype=np.int32), s)
    assert np.all(zero == 0)


def test_few_query_kernel_queries_before_the_cache():
    # len_b < Lq under the cached-decoding mask: the first Lq - len_b rows see no key
    s = spec(3, 4, 8, 300, 64, mask=TAIL | KP, Hkv=2)
    assert _path(s) == DECODE_PATH
    q, k, v, _ = gen.make_inputs(s, seed=33)
    lens = np.array([3, 0, 300], dtype=np.int32)
    out = run_gpu(q, k, v, lens, s)
    ref = oracle.mha_fwd(q, k, v, mask_kind=TAIL | KP, key_lengths=lens,
                         scale=gen.default_scale(64))
    compare(out, ref, "bf16")
    assert np.all(out[0, :, :5] == 0) and np.all(out[1] == 0)


@pytest.mark.parametrize("d", [64, 128])
def test_few_query_kernel_climbing_scores(d):
    # scores rising along the keys: the running maximum moves tile after tile
    # and the partial output held in tensor memory is rescaled; then falling
    rng = np.random.default_rng(34)
    B, H, Hkv, Lq, Lk = 2, 4, 1, 2, 1500
    q = np.abs(rng.normal(size=(B, H, Lq, d))) * 0.5 + 0.5
    ramp = (np.arange(Lk) / 64.0)[None, None, :, None] * (64.0 / d)
    k = ramp * (0.5 + 0.1 * rng.normal(size=(B, Hkv, Lk, d)))
    v = rng.normal(size=(B, Hkv, Lk, d))
    q, k, v = (gen.f64_to_bf16_bits(x) for x in (q, k, v))
    s = spec(B, H, Lq, Lk, d, mask=TAIL | KP, Hkv=Hkv)
    assert _path(s) == DECODE_PATH
    lens = np.array([Lk - 3, 700], dtype=np.int32)
    for kk, label in ((k, "climbing"), (np.ascontiguousarray(k[:, :, ::-1]), "falling")):
        out = run_gpu(q, kk, v, lens, s)
        ref = oracle.mha_fwd(q, kk, v, mask_kind=TAIL | KP, key_lengths=lens,
                             scale=gen.default_scale(d))
        compare(out, ref, "bf16", label=label)


@pytest.mark.parametrize("scale", [0.0, -0.3, 1.0])
def test_few_query_kernel_other_scales(scale):
    check_case(spec(3, 8, 1, 900, 64, mask=TAIL | KP, len_range=(1, 900), Hkv=2), seed=35,
               scale=scale)
    check_case(spec(2, 4, 4, 600, 128, mask=TAIL, Hkv=1, layout="bshd"), seed=35, scale=scale)


def test_few_query_kernel_deterministic_and_matches_repeated_heads():
    s = spec(6, 8, 1, 1000, 128, mask=TAIL | KP, len_range=(1, 1000), Hkv=2, layout="bshd")
    q, k, v, lens = gen.make_inputs(s, seed=36)
    a = run_gpu(q, k, v, lens, s)
    np.testing.assert_array_equal(a, run_gpu(q, k, v, lens, s))
    # sharing a key/value head among 4 query heads gives the same bits as
    # giving each its own copy
    rep = run_gpu(q, np.repeat(k, 4, axis=2), np.repeat(v, 4, axis=2), lens, dict(s, Hkv=8))
    np.testing.assert_array_equal(a, rep)


def test_decode_workload_full_size_all_rows():
    s = gen.WORKLOADS["decode_bf16_b256_h8_lk1024_d64"]
    assert _path(s) == DECODE_PATH
    check_case(s, label="decode full size")


def test_decode_gqa_workload_full_size_sampled_rows():
    s = gen.WORKLOADS["decode_gqa_bf16_b64_h32_kv8_lk8192_d128"]
    assert _path(s) == DECODE_PATH
    rng = np.random.default_rng(37)
    rows = np.array(sorted(set(rng.integers(0, s["B"] * s["H"], 256))), dtype=np.int64)
    check_case(s, rows=rows, label="decode gqa full size (sampled)")
