"""The bench's algorithmic work per launch, the numerator of every throughput
and roofline figure it reports: flops = 2 (d_k + d_v) per allowed (query, key)
pair, bytes = the Q rows that are not query padding, the K and V rows that are
not key padding, every output row and the lengths.  Checked against a brute
force over the mask definitions on small shapes and against the closed forms
of the full causal and unmasked workloads."""
import numpy as np
import pytest

import bench
import gen

C, KP, QP, CT = gen.MASK_CAUSAL, gen.MASK_KEY_PADDING, gen.MASK_QUERY_PADDING, gen.MASK_CAUSAL_TAIL


def brute(spec, lens):
    B, H, Lq, Lk, dk, dv = (spec[x] for x in ("B", "H", "Lq", "Lk", "dk", "dv"))
    Hkv = spec.get("Hkv", H)
    m = spec["mask"]
    esz = 4 if spec["dtype"] == "f32" else 2
    pairs = q_rows = kv_rows = 0
    for b in range(B):
        L = Lk if lens is None else min(max(int(lens[b]), 0), Lk)
        for i in range(Lq):
            if m & QP and i >= L:
                continue  # a padded query row: stored as zeros, never computed
            q_rows += H
            for j in range(Lk):
                allowed = not (m & C and j > i) and not (m & KP and j >= L) and \
                    not (m & CT and j > L - Lq + i)
                pairs += H if allowed else 0
        kv_rows += (L if m & KP else Lk) * Hkv
    nbytes = esz * (q_rows * dk + kv_rows * (dk + dv) + B * H * Lq * dv)
    if lens is not None and m & (KP | QP):
        nbytes += 4 * B
    return nbytes, 2 * (dk + dv) * pairs


CASES = [
    # (B, H, Hkv, Lq, Lk, d, dtype, mask, lengths)
    (3, 2, 2, 9, 9, 8, "bf16", 0, None),
    (3, 2, 2, 9, 9, 8, "bf16", C, None),
    (4, 2, 1, 7, 7, 8, "bf16", KP | QP, [0, 3, 7, 9]),
    (4, 2, 2, 5, 11, 16, "f32", KP, [1, 11, 4, 0]),
    (3, 4, 2, 6, 6, 8, "bf16", C | KP, [2, 6, 5]),
    (3, 4, 1, 2, 13, 8, "bf16", CT | KP, [1, 13, 7]),
    (2, 2, 2, 3, 10, 8, "bf16", CT, None),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "m%d_%s" % (c[7], c[6]))
def test_counts_match_brute_force(case):
    B, H, Hkv, Lq, Lk, d, dt, mask, lens = case
    spec = dict(B=B, H=H, Hkv=Hkv, Lq=Lq, Lk=Lk, dk=d, dv=d, dtype=dt, mask=mask)
    lens = np.array(lens, dtype=np.int32) if lens is not None else None
    assert bench.algorithmic(spec, lens) == brute(spec, lens)


def test_seeded_padded_workloads_match_brute_force():
    # the realised lengths of the padded workloads, on a few batch elements
    for name in ("enc_pad_bf16_b256_h8_l64_d64", "cross_pad_bf16_b64_h16_lq96_lk128_d64",
                 "decode_bf16_b256_h8_lk1024_d64"):
        spec = dict(gen.WORKLOADS[name])
        lo, hi = spec["len_range"]
        lens = gen.lengths(0, spec["B"], lo, hi)[:5]  # as the workload draws them
        spec["B"] = 5
        assert bench.algorithmic(spec, lens) == brute(spec, lens), name


def test_closed_forms_of_the_full_workloads():
    # causal: L (L + 1) / 2 allowed pairs per head; no padding: every row moves
    w = gen.WORKLOADS
    for name, B, H, L, d in (("dec_causal_bf16_b128_h8_l128_d64", 128, 8, 128, 64),
                             ("long_causal_bf16_b4_h16_l8192_d128", 4, 16, 8192, 128)):
        nbytes, flops = bench.algorithmic(w[name], None)
        assert flops == B * H * (L * (L + 1) // 2) * 2 * (2 * d)
        assert nbytes == 4 * B * H * L * d * 2
    nbytes, flops = bench.algorithmic(w["enc_f32_b2_h8_l32_d64"], None)
    assert flops == 2 * 8 * 32 * 32 * 2 * 128  # 4.19 MFLOP
    assert nbytes == 4 * 2 * 8 * 32 * 64 * 4  # 512 KiB
    assert bench.algorithmic(w["long_causal_bf16_b4_h16_l8192_d128"], None)[1] == \
        pytest.approx(1.0996e12, rel=1e-4)


@pytest.mark.parametrize("case", CASES)
def test_backward_flops_are_five_products_per_allowed_pair(case):
    # scores recomputed (2 d_k), dP (2 d_v), dV (2 d_v), dK (2 d_k), dQ (2 d_k)
    B, H, Hkv, Lq, Lk, d, dtype, mask, lens = case
    spec = dict(B=B, H=H, Hkv=Hkv, Lq=Lq, Lk=Lk, dk=d, dv=d, dtype=dtype, mask=mask)
    lens_a = None if lens is None else np.asarray(lens, dtype=np.int32)
    _, fwd = brute(spec, lens_a)
    pairs = fwd // (2 * (d + d))
    assert bench.backward_flops(spec, lens_a) == pairs * 2 * (3 * d + 2 * d)


def test_projection_kernel_name_follows_the_tiling_rule():
    # 128 x 256 tiles when K and N are multiples of 64 and N >= 256
    assert bench.linear_kernel_name(512, 512) == "linear_wide_kernel"
    assert bench.linear_kernel_name(512, 256) == "linear_wide_kernel"
    assert bench.linear_kernel_name(512, 192) == "linear_tc_kernel"
    assert bench.linear_kernel_name(200, 512) == "linear_tc_kernel"
    assert bench.linear_kernel_name(512, 320) == "linear_wide_kernel"
    assert bench.linear_kernel_name(512, 72) == "linear_tc_kernel"


def test_backward_kernel_names_follow_the_dispatch_rule():
    # the fused single-tile kernel (d 64, lengths <= 128): its storing form
    # <1> with the forward's statistics unless the mask is causal
    C, KP, TAIL = gen.MASK_CAUSAL, gen.MASK_KEY_PADDING, gen.MASK_CAUSAL_TAIL
    assert bench.bwd_kernel_names(64, 128, 128, C)[1] == "bwd_short_tc_kernel<0>"
    assert bench.bwd_kernel_names(64, 96, 128, KP)[1] == "bwd_short_tc_kernel<1>"
    assert bench.bwd_kernel_names(64, 16, 100, TAIL | KP)[1] == "bwd_short_tc_kernel<1>"
    assert bench.bwd_kernel_names(64, 64, 64, 0)[0] == "bwd_short_tc_kernel<1> (one launch)"
    for dk, Lq, Lk in ((128, 128, 128), (64, 129, 128), (64, 128, 8192)):
        assert bench.bwd_kernel_names(dk, Lq, Lk, C)[1].startswith("bwd_dkdv_tc_kernel")
    # the committed traffic record of each backward workload was taken on the
    # kernel that the bench's timed calls run
    import json
    import os
    with open(os.path.join(os.path.dirname(bench.__file__), "profiles", "traffic.json")) as f:
        records = json.load(f)
    for w, fwd in bench.BWD_WORKLOADS.items():
        s = gen.WORKLOADS[fwd]
        want = bench.bwd_kernel_names(s["dk"], s["Lq"], s["Lk"], s["mask"])[1].split(" ")[0]
        if w in records:
            got = records[w]["kernel_name"]
            assert got == want or got.startswith(want + "<"), (w, got, want)
