"""GPU parity of the backward pass (mha_bwd) against the fp64 oracle's
gradients (oracle.mha_bwd, pinned by finite differences).

The GPU side runs as a user would: the forward (mha_fwd_ex) gives `out`, then
mha_bwd takes q, k, v, out and the incoming gradient dout.  Errors are
measured against each gradient tensor's largest magnitude (the sums behind
dq and dk cancel -- each row's dS sums to zero -- so single elements can be far
smaller than the terms that formed them):

  fp32: max |err| <= 1e-4 * max|ref|
  bf16: max |err| <= 2e-2 * max|ref|, mean |err| <= 2e-3 * max|ref|
        (inputs, out and the stored gradients are bf16, relative 2^-9 each)

Gradients that are zero by the masks alone -- dq of rows that attend to
nothing, dk and dv of keys no row may read -- must be exactly zero.
"""
import numpy as np
import pytest

import gen
import oracle
from helpers import from_device, spec, to_device

pytestmark = pytest.mark.gpu

C, KP, QP, TAIL = gen.MASK_CAUSAL, gen.MASK_KEY_PADDING, gen.MASK_QUERY_PADDING, \
    gen.MASK_CAUSAL_TAIL
BWD_TOL = {"f32": dict(max=1e-4, mean=1e-4), "bf16": dict(max=2e-2, mean=2e-3)}


def run_bwd(s, seed, lens=None, scale=None, use_lse=False):
    """Forward then backward on the GPU; with ``use_lse`` the forward is
    mha_fwd_lse (its output must equal mha_fwd_ex's bit for bit) and the
    backward takes its row statistics."""
    import torch
    import transformer_head_scaled_mha_gb300 as mha
    q, k, v, glens = gen.make_inputs(s, seed=seed)
    lens = glens if lens is None else np.asarray(lens, dtype=np.int32)
    dout = gen.make_dout(s, seed=seed)
    dt, layout = s["dtype"], s.get("layout", "bhsd")
    scale = gen.default_scale(s["dk"]) if scale is None else scale
    kl = torch.from_numpy(lens).cuda() if lens is not None else None
    Q, K, V, DO = (to_device(a, dt) for a in (q, k, v, dout))
    out = mha.mha_fwd_ex(Q, K, V, layout=layout, mask_kind=s["mask"], key_lengths=kl, scale=scale)
    assert np.isfinite(gen.as_f64(from_device(out), dt)).all(), "forward output non-finite"
    lse = None
    if use_lse:
        out2, lse = mha.mha_fwd_lse(Q, K, V, layout=layout, mask_kind=s["mask"], key_lengths=kl,
                                    scale=scale)
        assert torch.equal(out2.view(torch.int16 if dt == "bf16" else torch.int32),
                           out.view(torch.int16 if dt == "bf16" else torch.int32))
    dq, dk, dv = mha.mha_bwd(Q, K, V, out, DO, layout=layout, mask_kind=s["mask"], key_lengths=kl,
                             scale=scale, lse=lse)
    torch.cuda.synchronize()
    assert mha.mha_debug_status() == mha.MHA_OK
    got = [gen.as_f64(from_device(t), dt) for t in (dq, dk, dv)]
    ref = oracle.mha_bwd(q, k, v, dout, mask_kind=s["mask"], key_lengths=lens, scale=scale,
                         layout=layout)
    return got, (ref, structural_zeros(s, lens))


def structural_zeros(s, lens):
    """Boolean masks (dq, dk, dv) of the gradients that the masks alone make zero."""
    B, H, Hkv, Lq, Lk, m = s["B"], s["H"], s["Hkv"], s["Lq"], s["Lk"], s["mask"]
    i = np.arange(Lq)[:, None]
    j = np.arange(Lk)[None, :]
    ok = np.ones((B, Lq, Lk), dtype=bool)
    for b in range(B):
        ln = Lk if lens is None else int(np.clip(lens[b], 0, Lk))
        a = np.ones((Lq, Lk), dtype=bool)
        if m & QP:
            a &= i < ln
        if m & C:
            a &= j <= i
        if m & KP:
            a &= j < ln
        if m & TAIL:
            a &= j <= ln - Lq + i
        ok[b] = a
    row_dead = ~ok.any(axis=2)  # [B, Lq]
    key_dead = ~ok.any(axis=1)  # [B, Lk]
    bshd = s.get("layout", "bhsd") == "bshd"
    zq = np.broadcast_to(row_dead[:, :, None, None] if bshd else row_dead[:, None, :, None],
                         (B, Lq, H, s["dk"]) if bshd else (B, H, Lq, s["dk"]))
    shape_k = (B, Lk, Hkv, s["dk"]) if bshd else (B, Hkv, Lk, s["dk"])
    zk = np.broadcast_to(key_dead[:, :, None, None] if bshd else key_dead[:, None, :, None],
                         shape_k)
    zv = np.broadcast_to(key_dead[:, :, None, None] if bshd else key_dead[:, None, :, None],
                         shape_k[:-1] + (s["dv"],))
    return zq, zk, zv


def compare_grads(got, ref_zero, dtype, label=""):
    ref, zeros = ref_zero
    tol = BWD_TOL[dtype]
    stats = []
    for g, r, z, name in zip(got, ref, zeros, ("dq", "dk", "dv")):
        assert np.isfinite(g).all(), "%s %s: non-finite" % (label, name)
        mag = float(np.abs(r).max()) if r.size else 0.0
        err = np.abs(g - r)
        if mag == 0.0:
            assert np.all(g == 0), "%s %s: reference is all zero" % (label, name)
            continue
        mx, mean = float(err.max()) / mag, float(err.mean()) / mag
        stats.append((name, mx, mean))
        assert mx <= tol["max"], "%s %s: max|err| %.3g of max|ref| > %.3g" % (label, name, mx,
                                                                             tol["max"])
        assert mean <= tol["mean"], "%s %s: mean|err| %.3g of max|ref|" % (label, name, mean)
        assert np.all(g[z] == 0), "%s %s: masked-out gradients not zero" % (label, name)
    return stats


def _id(s):
    return "B%dH%dKV%dLq%dLk%dd%d_%s_m%d_%s" % (s["B"], s["H"], s["Hkv"], s["Lq"], s["Lk"],
                                                s["dk"], s["dtype"], s["mask"], s["layout"])


CASES = [
    spec(2, 2, 32, 32, 64, "f32"),
    spec(2, 3, 45, 77, 100, "f32", mask=KP, len_range=(0, 77)),
    spec(2, 2, 50, 50, 17, "f32", mask=C, Hkv=1, layout="bshd"),
    spec(2, 2, 40, 40, 128, "f32", mask=KP | QP, len_range=(0, 40)),
    spec(2, 4, 6, 90, 64, "f32", mask=TAIL | KP, len_range=(0, 90), Hkv=2),
    spec(4, 2, 64, 64, 64, mask=KP | QP, len_range=(0, 64)),
    spec(2, 2, 128, 128, 64, mask=C),
    spec(2, 4, 96, 128, 64, mask=KP, len_range=(16, 128), Hkv=2, layout="bshd"),
    spec(1, 2, 300, 300, 128, mask=C, amp=0.5),
    spec(2, 2, 200, 333, 64, mask=KP, len_range=(0, 333)),
    spec(1, 4, 257, 257, 128, mask=C | KP, len_range=(100, 257), Hkv=1, layout="bshd"),
    spec(3, 2, 1, 500, 64, mask=TAIL | KP, len_range=(1, 500)),
    # short tiles packed several (batch, head) pairs to a tile, heads past
    # the last one in a tile's final group
    spec(3, 5, 20, 20, 64, mask=KP | QP, len_range=(0, 20)),
    spec(2, 16, 8, 8, 64, mask=C),
    spec(2, 3, 50, 33, 64, mask=KP, len_range=(1, 33), layout="bshd"),
    spec(4, 8, 64, 64, 64, mask=KP | QP, len_range=(8, 64), layout="bshd"),
    # single-tile decoding against a short padded cache; no mask (pairs packed)
    spec(2, 4, 16, 100, 64, mask=TAIL | KP, len_range=(20, 100)),
    spec(3, 4, 40, 40, 64),
    # several query and key tiles with shared key/value heads
    spec(2, 4, 640, 640, 128, mask=C, amp=0.5, Hkv=2, layout="bshd"),
    spec(2, 6, 333, 555, 64, mask=KP, len_range=(100, 555), Hkv=3),
    spec(2, 4, 260, 700, 64, mask=TAIL | KP, len_range=(300, 700), Hkv=1, layout="bshd"),
]


@pytest.mark.parametrize("s", CASES, ids=_id)
def test_backward_parity(s):
    got, ref = run_bwd(s, seed=41)
    compare_grads(got, ref, s["dtype"], label=_id(s))


@pytest.mark.parametrize("s", CASES, ids=_id)
def test_backward_parity_with_forward_lse(s):
    # mha_bwd_lse: the forward's statistics in place of the statistics pass
    got, ref = run_bwd(s, seed=41, use_lse=True)
    compare_grads(got, ref, s["dtype"], label=_id(s) + " lse")


def test_backward_with_forward_lse_padding_edges():
    s = spec(4, 2, 64, 64, 64, mask=KP | QP, layout="bshd", Hkv=1)
    got, ref = run_bwd(s, seed=42, lens=[0, 1, 64, 33], use_lse=True)
    compare_grads(got, ref, "bf16", label="padding edges lse")
    dq, dk, dv = got
    assert np.all(dq[0] == 0) and np.all(dk[0] == 0) and np.all(dv[0] == 0)


def test_backward_padding_edges():
    # empty sequences and a sequence of one key among full ones
    s = spec(4, 2, 64, 64, 64, mask=KP | QP, layout="bshd", Hkv=1)
    got, ref = run_bwd(s, seed=42, lens=[0, 1, 64, 33])
    compare_grads(got, ref, "bf16", label="padding edges")
    dq, dk, dv = got
    assert np.all(dq[0] == 0) and np.all(dk[0] == 0) and np.all(dv[0] == 0)
    assert np.all(dq[1, 1:] == 0) and np.all(dk[1, 1:] == 0)


@pytest.mark.parametrize("scale", [0.0, -0.3])
def test_backward_other_scales(scale):
    for s in (spec(2, 2, 64, 64, 64, mask=C), spec(2, 2, 40, 40, 64, "f32", mask=KP | QP,
                                                      len_range=(1, 40))):
        got, ref = run_bwd(s, seed=43, scale=scale)
        compare_grads(got, ref, s["dtype"], label="scale %g" % scale)


def test_backward_no_keys_gives_zero_gradients():
    import torch
    import transformer_head_scaled_mha_gb300 as mha
    q = torch.randn(2, 2, 8, 64, device="cuda").bfloat16()
    k = torch.empty(2, 2, 0, 64, device="cuda", dtype=torch.bfloat16)
    out = torch.zeros_like(q)
    dq, dk, dv = mha.mha_bwd(q, k, k, out, torch.randn_like(q))
    torch.cuda.synchronize()
    assert torch.all(dq == 0) and dk.numel() == 0 and dv.numel() == 0


def test_backward_deterministic():
    s = spec(2, 4, 128, 128, 64, mask=C, Hkv=2)
    a, _ = run_bwd(s, seed=44)
    b, _ = run_bwd(s, seed=44)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_backward_rejects_small_workspace():
    import torch
    import transformer_head_scaled_mha_gb300 as mha
    q = torch.randn(1, 2, 16, 64, device="cuda").bfloat16()
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(mha.MhaError):
        mha.mha_bwd(q, q, q, q.clone(), q.clone(), workspace=ws)


def test_backward_long_causal_full_size_sampled():
    # the long causal workload at full size; rows [L-128, L) of a head give
    # its dq exactly and, under the causal mask, the whole dk and dv of keys
    # [L-128, L); rows [0, 128) give their dq exactly
    import torch
    import transformer_head_scaled_mha_gb300 as mha
    s = gen.WORKLOADS["long_causal_bf16_b4_h16_l8192_d128"]
    L, B, H = s["Lq"], s["B"], s["H"]
    q, k, v, _ = gen.make_inputs(s, seed=45)
    dout = gen.make_dout(s, seed=45)
    scale = gen.default_scale(s["dk"])
    Q, K, V, DO = (to_device(a, "bf16") for a in (q, k, v, dout))
    out = mha.mha_fwd(Q, K, V, mask_kind=C, scale=scale)
    dq, dk, dv = mha.mha_bwd(Q, K, V, out, DO, mask_kind=C, scale=scale)
    torch.cuda.synchronize()
    assert mha.mha_debug_status() == mha.MHA_OK
    got = [gen.as_f64(from_device(t), "bf16") for t in (dq, dk, dv)]
    del Q, K, V, DO, out, dq, dk, dv
    units = [0, 17, 38, 63]
    ref_hi = oracle.mha_bwd(q, k, v, dout, mask_kind=C, scale=scale, units=units,
                            rows=(L - 128, L))
    ref_lo = oracle.mha_bwd(q, k, v, dout, mask_kind=C, scale=scale, units=units, rows=(0, 128))
    for u in units:
        b, h = divmod(u, H)
        pieces = [(got[0][b, h, L - 128:], ref_hi[0][b, h, L - 128:], "dq last rows"),
                  (got[0][b, h, :128], ref_lo[0][b, h, :128], "dq first rows"),
                  (got[1][b, h, L - 128:], ref_hi[1][b, h, L - 128:], "dk last keys"),
                  (got[2][b, h, L - 128:], ref_hi[2][b, h, L - 128:], "dv last keys")]
        for g, r, name in pieces:
            mag = float(np.abs(r).max())
            err = np.abs(g - r)
            assert err.max() <= 2e-2 * mag and err.mean() <= 2e-3 * mag, (u, name, err.max(), mag)
