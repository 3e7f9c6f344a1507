"""The C ABI: the library loads, exports what include/mha.h declares, and
rejects bad arguments before touching the GPU (these calls never reach CUDA)."""
import ctypes
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def mha():
    import __graft_entry__
    __graft_entry__._load_build_module().build()
    import transformer_head_scaled_mha_gb300 as m
    return m


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mha.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mha_\w+)\s*\(", src)))


def test_header_declares_the_entry_points():
    assert declared_functions() == sorted(
        ["mha_fwd", "mha_fwd_ex", "mha_fwd_lse", "mha_bwd_lse", "mha_linear_fwd",
         "mha_sublayer_workspace_size",
         "mha_sublayer_fwd", "mha_sublayer_fwd_static", "mha_bwd_workspace_size", "mha_bwd",
         "mha_fwd_path", "mha_fwd_path_ex",
         "mha_status_string", "mha_debug_status", "mha_debug_set_wait",
         "mha_version"])


def test_library_exports_every_declared_symbol(mha):
    lib = ctypes.CDLL(mha.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(mha.mha.EXPORTED) == set(declared_functions())


def test_status_strings(mha):
    assert mha.mha_status_string(0) == "ok"
    assert "invalid" in mha.mha_status_string(1)
    assert "unsupported" in mha.mha_status_string(2)
    assert mha.mha_status_string(99) == "unknown status"
    assert mha.mha_version() >= 100


def test_debug_wait_hook_rejects_unknown_stall_bits(mha):
    assert mha.mha_debug_set_wait(0, 4) == mha.MHA_ERR_INVALID_ARGUMENT
    assert mha.mha_debug_set_wait(0, 0) == mha.MHA_OK  # the defaults


def test_path_selection(mha):
    P = mha.mha_fwd_path
    assert P(2, 8, 32, 32, 64, 64, 0, 0) == 1  # fp32
    assert P(256, 8, 64, 64, 64, 64, 6, 1) == 2  # packed short
    assert P(128, 8, 128, 128, 64, 64, 1, 1) == 2
    assert P(64, 16, 96, 128, 64, 64, 2, 1) == 2
    assert P(4, 16, 8192, 8192, 128, 128, 1, 1) == 3  # long
    assert P(2, 2, 129, 129, 64, 64, 1, 1) == 3
    assert P(2, 2, 64, 64, 128, 128, 0, 1) == 3
    assert P(0, 2, 64, 64, 64, 64, 0, 1) == 0  # empty
    assert P(2, 2, 64, 0, 64, 64, 0, 1) == 4  # no keys: zero fill
    assert P(2, 2, 64, 64, 96, 96, 0, 1) == -2  # bf16 d must be 64 or 128
    assert P(2, 2, 64, 64, 64, 128, 0, 1) == -2
    assert P(2, 2, 64, 64, 129, 64, 0, 0) == -2
    assert P(2, 2, 64, 65, 64, 64, 1, 1) == -1  # causal needs Lq == Lk
    assert P(2, 2, 64, 65, 64, 64, 4, 1) == -1  # query padding needs Lq == Lk
    assert P(2, 2, 1, 4096, 128, 128, 8 | 2, 1) == 5  # cached decoding: few query rows
    assert P(2, 2, 16, 4096, 64, 64, 8, 1) == 5
    assert P(2, 2, 1, 129, 64, 64, 0, 1) == 5
    assert P(2, 2, 1, 100, 128, 128, 2, 1) == 5
    assert P(2, 2, 17, 4096, 64, 64, 8, 1) == 3  # more than 16 rows: long kernel
    assert P(2, 2, 1, 100, 64, 64, 8, 1) == 2  # d = 64, Lk <= 128: packed kernel
    assert P(2, 2, 4, 4096, 128, 128, 8 | 2, 0) == 1  # fp32
    assert P(2, 2, 64, 64, 64, 64, 8 | 1, 1) == -1  # not with CAUSAL
    assert P(2, 2, 64, 64, 64, 64, 8 | 4, 1) == -1  # not with QUERY_PADDING
    assert P(2, 2, 64, 64, 64, 64, 16, 1) == -1  # unknown mask bit
    assert P(-1, 2, 64, 64, 64, 64, 0, 1) == -1
    assert P(2, 2, 64, 64, 0, 64, 0, 1) == -1
    assert P(2, 2, 64, 64, 64, 64, 0, 7) == -1  # unknown dtype


def test_path_selection_with_shared_heads(mha):
    # the few-query kernel takes (H / H_kv) * Lq <= 16 query rows per key/value head
    PX = mha.mha_fwd_path_ex
    assert PX(64, 32, 8, 1, 8192, 128, 128, 8 | 2, 1) == 5  # 4 rows
    assert PX(2, 32, 2, 1, 8192, 128, 128, 8 | 2, 1) == 5  # 16 rows
    assert PX(2, 32, 1, 1, 8192, 128, 128, 8 | 2, 1) == 3  # 32 rows: long kernel
    assert PX(2, 8, 2, 4, 1000, 64, 64, 8, 1) == 5
    assert PX(2, 8, 2, 5, 1000, 64, 64, 8, 1) == 3
    assert PX(2, 8, 8, 1, 1000, 64, 64, 1, 1) == -1  # causal needs Lq == Lk
    assert PX(2, 8, 3, 1, 1000, 64, 64, 0, 1) == -1  # H_kv must divide H
    assert PX(2, 8, 0, 1, 1000, 64, 64, 0, 1) == -1
    for args in [(2, 8, 1000, 1000, 64, 64, 1, 1), (256, 8, 1, 1024, 64, 64, 10, 1),
                 (2, 2, 64, 64, 96, 96, 0, 1)]:
        B, H = args[:2]
        assert PX(B, H, H, *args[2:]) == mha.mha_fwd_path(*args)


FAKE = 0x7F0000000000  # never dereferenced: every call below fails validation first


def call(mha, q=FAKE, k=FAKE + (1 << 24), v=FAKE + (2 << 24), out=FAKE + (3 << 24), B=2, H=2,
         Lq=64, Lk=64, dk=64, dv=64, mask=0, kl=None, scale=0.125, dtype=1):
    return mha.lib.mha_fwd(q, k, v, out, B, H, Lq, Lk, dk, dv, mask, kl, scale, dtype, None)


def test_rejects_before_launch(mha):
    E_ARG, E_UNS = mha.MHA_ERR_INVALID_ARGUMENT, mha.MHA_ERR_UNSUPPORTED
    assert call(mha, B=-1) == E_ARG
    assert call(mha, dk=0) == E_ARG
    assert call(mha, mask=1, Lk=65) == E_ARG
    assert call(mha, mask=2) == E_ARG  # key_lengths missing
    assert call(mha, mask=4) == E_ARG
    assert call(mha, q=None) == E_ARG
    assert call(mha, out=None) == E_ARG
    assert call(mha, k=None) == E_ARG
    assert call(mha, q=FAKE + 8) == E_ARG  # not 16-byte aligned
    assert call(mha, out=FAKE + 4096) == E_ARG  # out overlaps q
    assert call(mha, out=FAKE + (2 << 24) + 64) == E_ARG  # out overlaps v
    assert call(mha, mask=2, kl=FAKE + (3 << 24) + 128) == E_ARG  # out overlaps key_lengths
    assert call(mha, mask=2, kl=FAKE + (5 << 24) + 2) == E_ARG  # int32 lengths not 4-byte aligned
    assert call(mha, mask=4, kl=FAKE + (5 << 24) + 1) == E_ARG
    assert call(mha, scale=math.inf) == E_ARG
    assert call(mha, scale=math.nan) == E_ARG
    assert call(mha, dtype=3) == E_ARG
    assert call(mha, dk=96, dv=96) == E_UNS
    assert call(mha, dk=64, dv=128) == E_UNS
    assert call(mha, dtype=0, dk=200) == E_UNS


def call_ex(mha, q=FAKE, k=FAKE + (1 << 24), v=FAKE + (2 << 24), out=FAKE + (3 << 24), B=2,
            H=4, Hkv=2, Lq=64, Lk=64, dk=64, dv=64, layout=0, mask=0, kl=None, scale=0.125,
            dtype=1):
    return mha.lib.mha_fwd_ex(q, k, v, out, B, H, Hkv, Lq, Lk, dk, dv, layout, mask, kl, scale,
                              dtype, None)


def test_ex_rejects_before_launch(mha):
    E_ARG, E_UNS = mha.MHA_ERR_INVALID_ARGUMENT, mha.MHA_ERR_UNSUPPORTED
    assert call_ex(mha, Hkv=3) == E_ARG  # does not divide H
    assert call_ex(mha, Hkv=0) == E_ARG
    assert call_ex(mha, Hkv=-2) == E_ARG
    assert call_ex(mha, Hkv=8) == E_ARG  # more key/value heads than query heads
    assert call_ex(mha, layout=2) == E_ARG
    assert call_ex(mha, layout=-1) == E_ARG
    assert call_ex(mha, layout=1, mask=2) == E_ARG  # key_lengths missing
    assert call_ex(mha, layout=1, q=FAKE + 8) == E_ARG
    assert call_ex(mha, layout=1, dk=96, dv=96) == E_UNS
    # k holds H_kv heads: an out over its last 16 bytes is caught
    k_bytes = 2 * 2 * 64 * 64 * 2
    assert call_ex(mha, out=FAKE + (1 << 24) + k_bytes - 16) == E_ARG
    assert call_ex(mha, B=0) == mha.MHA_OK
    assert call_ex(mha, B=0, Hkv=3) == E_ARG  # arguments are checked even when empty
    assert call_ex(mha, H=0, Hkv=0, B=2) == mha.MHA_OK


def test_empty_problem_returns_ok_without_device(mha):
    # B*H*Lq == 0 enqueues nothing, so it succeeds even without a GPU
    assert call(mha, B=0) == mha.MHA_OK
    assert call(mha, Lq=0, q=None, out=None) == mha.MHA_OK


def test_binding_refuses_cpu_tensors(mha):
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        mha.mha_fwd(q, q, q)


def test_lse_entry_points_reject_before_launch(mha):
    E_ARG = mha.MHA_ERR_INVALID_ARGUMENT
    q, k, v, out = FAKE, FAKE + (1 << 24), FAKE + (2 << 24), FAKE + (3 << 24)
    lse = FAKE + (4 << 24)

    def fwd(lse_=lse, B=2, mask=0, kl=None):
        return mha.lib.mha_fwd_lse(q, k, v, out, lse_, B, 4, 2, 64, 64, 64, 64, 0, mask, kl,
                                   0.125, 1, None)
    assert fwd(lse_=None) == E_ARG  # the statistics are this call's purpose
    assert fwd(lse_=lse + 2) == E_ARG  # not 4-byte aligned
    assert fwd(lse_=out + 64) == E_ARG  # overlaps out
    assert fwd(lse_=q + 128) == E_ARG  # overlaps q
    assert fwd(lse_=None, B=0) == mha.MHA_OK  # empty
    ws_n = mha.mha_bwd_workspace_size(2, 4, 64)
    p = [FAKE + (i << 24) for i in range(11)]

    def bwd(lse_=p[10], ws=p[8]):
        return mha.lib.mha_bwd_lse(p[0], p[1], p[2], p[3], p[4], lse_, p[5], p[6], p[7], 2, 4, 2,
                                   64, 64, 64, 64, 0, 0, None, 0.125, 1, ws, ws_n, None)
    assert bwd(lse_=None) == E_ARG
    assert bwd(lse_=p[10] + 1) == E_ARG  # not 4-byte aligned
    assert bwd(lse_=p[5] + 64) == E_ARG  # inside dq
    assert bwd(lse_=p[8] + 64) == E_ARG  # inside the workspace


def test_linear_rejects_before_launch(mha):
    E_ARG, E_UNS = mha.MHA_ERR_INVALID_ARGUMENT, mha.MHA_ERR_UNSUPPORTED
    L = mha.lib.mha_linear_fwd
    x, w, y = FAKE, FAKE + (1 << 24), FAKE + (2 << 24)
    assert L(x, w, None, y, -1, 512, 512, 1, None) == E_ARG
    assert L(x, w, None, y, 64, 0, 512, 1, None) == E_ARG
    assert L(x, w, None, y, 64, 512, 512, 0, None) == E_UNS  # fp32
    assert L(x, w, None, y, 64, 500, 512, 1, None) == E_UNS  # K not a multiple of 8
    assert L(x, w, None, y, 64, 512, 100, 1, None) == E_UNS
    assert L(x + 8, w, None, y, 64, 512, 512, 1, None) == E_ARG  # alignment
    assert L(x, w, FAKE + (3 << 24) + 1, y, 64, 512, 512, 1, None) == E_ARG
    assert L(x, w, None, x + 4096, 64, 512, 512, 1, None) == E_ARG  # y overlaps x
    assert L(x, w, None, y, 0, 512, 512, 1, None) == mha.MHA_OK  # empty: nothing to do


def test_sublayer_workspace_size(mha):
    n = mha.mha_sublayer_workspace_size(2, 64, 64, 512, 8, 8, 64, 64)
    assert n == 4 * 2 * 64 * 512 * 2
    assert mha.mha_sublayer_workspace_size(2, 64, 96, 512, 8, 2, 64, 64) == \
        2 * 64 * 512 * 2 * 2 + 2 * 2 * 96 * 128 * 2
    assert mha.mha_sublayer_workspace_size(-1, 64, 64, 512, 8, 8, 64, 64) == 0


def test_sublayer_rejects_before_launch(mha):
    E_ARG, E_UNS = mha.MHA_ERR_INVALID_ARGUMENT, mha.MHA_ERR_UNSUPPORTED
    S_ = mha.lib.mha_sublayer_fwd
    ws_n = mha.mha_sublayer_workspace_size(2, 64, 64, 512, 8, 8, 64, 64)
    p = [FAKE + (i << 24) for i in range(12)]
    x, mem, out, wq, wk, wv, wo, ws = p[0], p[1], p[2], p[3], p[4], p[5], p[6], p[7]

    def call(B=2, T=64, S=64, d=512, H=8, Hkv=8, dk=64, dv=64, mask=0, kl=None, scale=0.125,
             dtype=1, mem_=mem, work=ws, work_n=ws_n):
        return S_(x, mem_, out, wq, wk, wv, wo, None, None, None, None, B, T, S, d, H, Hkv, dk,
                  dv, mask, kl, scale, dtype, work, work_n, None)
    assert call(mem_=None, S=32) == E_ARG  # self-attention needs S == T
    assert call(H=8, Hkv=3) == E_ARG
    assert call(dtype=0) == E_UNS
    assert call(dk=96, dv=96) == E_UNS
    assert call(d=500) == E_UNS
    assert call(mask=2) == E_ARG  # key lengths missing
    assert call(mask=1, S=32) == E_ARG  # causal needs T == S
    assert call(work=None) == E_ARG
    assert call(work_n=ws_n - 1) == E_ARG
    assert call(work=ws + 64) == E_ARG  # workspace alignment
    assert call(work=out) == E_ARG  # workspace overlaps out
    assert call(scale=math.nan) == E_ARG
    assert call(mask=2, kl=ws + 512) == E_ARG  # lengths inside the workspace
    assert call(mask=2, kl=p[9] + 2) == E_ARG  # lengths not 4-byte aligned
    # H d_k past INT_MAX: rejected, not wrapped to a small projection width
    big = (1 << 26) + 1
    assert call(H=big, Hkv=big, work_n=mha.mha_sublayer_workspace_size(
        2, 64, 64, 512, big, big, 64, 64)) == E_UNS
    assert call(H=big, Hkv=1, work_n=1 << 62) == E_UNS
    assert call(B=0) == mha.MHA_OK


def test_static_sublayer_rejects_shapes_beyond_its_scratch(mha):
    # 64 MiB of static scratch: the Transformer-base encoder sublayer at
    # B=256, T=64 needs exactly that; one more batch element does not fit
    S_ = mha.lib.mha_sublayer_fwd_static
    p = [FAKE + (i << 24) for i in range(12)]
    call = lambda B: S_(p[0], None, p[2], p[3], p[4], p[5], p[6], None, None, None, None, B, 64,
                        64, 512, 8, 8, 64, 64, 0, None, 0.125, 1, None)
    assert mha.mha_sublayer_workspace_size(256, 64, 64, 512, 8, 8, 64, 64) == 64 << 20
    assert call(257) == mha.MHA_ERR_UNSUPPORTED
    assert call(-1) == mha.MHA_ERR_INVALID_ARGUMENT
    assert call(0) == mha.MHA_OK


def test_bwd_workspace_size(mha):
    # two fp32 values per query row, each part rounded up to 256 bytes
    assert mha.mha_bwd_workspace_size(2, 4, 64) == 2 * (2 * 4 * 64 * 4)
    assert mha.mha_bwd_workspace_size(1, 1, 3) == 2 * 256
    assert mha.mha_bwd_workspace_size(0, 4, 64) == 0
    assert mha.mha_bwd_workspace_size(2, 4, -1) == 0


def test_bwd_rejects_before_launch(mha):
    E_ARG, E_UNS = mha.MHA_ERR_INVALID_ARGUMENT, mha.MHA_ERR_UNSUPPORTED
    p = [FAKE + (i << 24) for i in range(10)]
    ws_n = mha.mha_bwd_workspace_size(2, 4, 64)

    def call(q=p[0], k=p[1], v=p[2], out=p[3], dout=p[4], dq=p[5], dk=p[6], dv=p[7], B=2, H=4,
             Hkv=2, Lq=64, Lk=64, d=64, layout=0, mask=0, kl=None, scale=0.125, dtype=1,
             ws=p[8], ws_n=ws_n):
        return mha.lib.mha_bwd(q, k, v, out, dout, dq, dk, dv, B, H, Hkv, Lq, Lk, d, d, layout,
                               mask, kl, scale, dtype, ws, ws_n, None)
    k_bytes = 2 * 2 * 64 * 64 * 2
    assert call(layout=2) == E_ARG
    assert call(scale=math.inf) == E_ARG
    assert call(mask=2) == E_ARG  # key lengths missing
    assert call(mask=1, Lk=65) == E_ARG  # causal needs Lq == Lk
    assert call(Hkv=3) == E_ARG  # does not divide H
    assert call(dtype=3) == E_ARG
    assert call(d=96) == E_UNS
    assert call(q=p[0] + 8) == E_ARG  # not 16-byte aligned
    assert call(dout=None) == E_ARG
    assert call(dq=None) == E_ARG
    assert call(dv=p[7] + 8) == E_ARG
    assert call(ws=None) == E_ARG
    assert call(ws_n=ws_n - 1) == E_ARG
    assert call(ws=p[8] + 16) == E_ARG  # workspace is 256-byte aligned
    assert call(dq=p[0] + 4096) == E_ARG  # dq overlaps q
    assert call(dk=p[7] - k_bytes + 16) == E_ARG  # dk overlaps dv
    assert call(dv=p[4] + 64) == E_ARG  # dv overlaps dout
    assert call(ws=p[3] + 1024) == E_ARG  # workspace overlaps out
    assert call(mask=2, kl=p[5] + 64) == E_ARG  # lengths inside dq
    assert call(mask=2, kl=p[8] + 64) == E_ARG  # lengths inside the workspace
    assert call(mask=2, kl=p[9] + 2) == E_ARG  # lengths not 4-byte aligned
    assert call(B=0) == mha.MHA_OK  # empty: nothing to do


class FakeCudaTensor:
    """Stands in for a CUDA tensor in the bindings' argument checks, which read
    only these attributes (no GPU needed; nothing is dereferenced)."""

    def __init__(self, shape, dtype="bf16", device="cuda:0", contiguous=True, ptr=FAKE):
        import torch
        self.shape = tuple(shape)
        self.dtype = {"bf16": torch.bfloat16, "f32": torch.float32, "i32": torch.int32,
                      "u8": torch.uint8}[dtype]
        self.device = torch.device(device)
        self.is_cuda = self.device.type == "cuda"
        self._contiguous, self._ptr = contiguous, ptr

    def dim(self):
        return len(self.shape)

    def is_contiguous(self):
        return self._contiguous

    def data_ptr(self):
        return self._ptr

    def numel(self):
        return math.prod(self.shape)

    def element_size(self):
        return self.dtype.itemsize


def test_sublayer_binding_checks_every_tensor_against_the_dimensions(mha):
    pytest.importorskip("torch")
    F = FakeCudaTensor
    B, T, S, d, H, Hkv, dk = 2, 16, 24, 128, 2, 1, 64

    def args(**over):
        a = dict(x=F((B, T, d)), w_q=F((d, H * dk)), w_k=F((d, Hkv * dk)), w_v=F((d, Hkv * dk)),
                 w_o=F((H * dk, d)), b_q=F((H * dk,)), b_k=F((Hkv * dk,)), b_v=F((Hkv * dk,)),
                 b_o=F((d,)), mem=F((B, S, d)), H=H, H_kv=Hkv, key_lengths=F((B,), "i32"),
                 scale=None, out=F((B, T, d)))
        a.update(over)
        return a
    out, dims, kl, scale, mem_ptr = mha.mha._sublayer_marshal(**args())
    assert dims == (B, T, S, d, H, Hkv, dk, dk)
    assert kl == FAKE and mem_ptr == FAKE and scale == pytest.approx(dk ** -0.5)
    bad = [dict(w_q=F((d + 8, H * dk))), dict(w_k=F((d, H * dk))), dict(w_o=F((H * dk, d + 8))),
           dict(b_o=F((d + 8,))), dict(b_q=F((dk,))), dict(mem=F((B, S, d + 8))),
           dict(mem=F((B + 1, S, d))), dict(out=F((B, T, d + 8))), dict(out=F((B, T, d), "f32")),
           dict(w_v=F((d, Hkv * dk), device="cuda:1")), dict(out=F((B, T, d), device="cuda:1")),
           dict(key_lengths=F((B,), "i32", device="cuda:1")),
           dict(key_lengths=F((B,), "i32", contiguous=False)), dict(key_lengths=F((B + 1,), "i32")),
           dict(x=F((B, T, d), device="cpu")), dict(H=3), dict(H=0)]
    for over in bad:
        with pytest.raises(ValueError):
            mha.mha._sublayer_marshal(**args(**over))
    # self-attention: no memory tensor, S = T
    assert mha.mha._sublayer_marshal(**args(mem=None))[1][2] == T
    assert mha.mha._workspace_bytes(F((100,), "f32"), F((1,)).device) == 400
    with pytest.raises(ValueError):
        mha.mha._workspace_bytes(F((100,), "u8", device="cuda:1"), F((1,)).device)


def test_attention_binding_checks_devices_and_lengths(mha):
    pytest.importorskip("torch")
    F = FakeCudaTensor
    q, k, v, out = F((2, 4, 8, 64)), F((2, 2, 8, 64)), F((2, 2, 8, 64)), F((2, 4, 8, 64))
    res = mha.mha._marshal(q, k, v, out, F((2,), "i32"), None, "bhsd")
    assert res[1] == (2, 4, 2, 8, 8, 64, 64) and res[2] == FAKE
    for bad in (dict(k=F((2, 2, 8, 64), device="cuda:1")), dict(out=F((2, 4, 8, 64), device="cuda:1")),
                dict(kl=F((2,), "i32", device="cuda:1")), dict(kl=F((2,), "i32", contiguous=False)),
                dict(out=F((2, 4, 8, 32)))):
        a = dict(q=q, k=k, v=v, out=out, kl=F((2,), "i32"))
        a.update(bad)
        with pytest.raises(ValueError):
            mha.mha._marshal(a["q"], a["k"], a["v"], a["out"], a["kl"], None, "bhsd")


def test_linear_binding_checks_devices(mha):
    pytest.importorskip("torch")
    F = FakeCudaTensor
    x, w = F((4, 16, 64)), F((64, 32))
    for kw in (dict(w=F((64, 32), device="cuda:1")), dict(b=F((32,), device="cuda:1")),
               dict(out=F((4, 16, 32), device="cuda:1")), dict(b=F((16,))), dict(w=F((48, 32)))):
        a = dict(x=x, w=w)
        a.update(kw)
        with pytest.raises(ValueError):
            mha.mha_linear_fwd(a.pop("x"), a.pop("w"), **a)


class _RecordingLib:
    """Takes the place of the loaded library: records each call's arguments."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def fn(*args):
            self.calls.append((name, args))
            return 0
        return fn


def test_bindings_pass_each_entry_point_its_declared_arguments(mha, monkeypatch):
    torch = pytest.importorskip("torch")
    import contextlib
    F = FakeCudaTensor
    real = mha.mha.lib
    rec = _RecordingLib()
    monkeypatch.setattr(mha.mha, "lib", rec)
    monkeypatch.setattr(torch.cuda, "device", lambda d: contextlib.nullcontext())
    kl = F((2,), "i32")
    q, k, v, o = F((2, 4, 8, 64)), F((2, 2, 8, 64)), F((2, 2, 8, 64)), F((2, 4, 8, 64))
    q4 = F((2, 4, 8, 64))
    mha.mha.mha_fwd(q, q4, q4, out=o, mask_kind=2, key_lengths=kl, stream=0)
    mha.mha.mha_fwd_ex(q, k, v, out=o, mask_kind=2, key_lengths=kl, stream=0)
    mha.mha.mha_bwd(q, k, v, o, F((2, 4, 8, 64)), mask_kind=2, key_lengths=kl, stream=0,
                    workspace=F((4096,), "u8"), dq=F((2, 4, 8, 64)), dk=F((2, 2, 8, 64)),
                    dv=F((2, 2, 8, 64)))
    mha.mha.mha_fwd_lse(q, k, v, out=o, lse=F((2, 4, 8), "f32"), mask_kind=2, key_lengths=kl,
                        stream=0)
    mha.mha.mha_bwd(q, k, v, o, F((2, 4, 8, 64)), mask_kind=2, key_lengths=kl, stream=0,
                    workspace=F((4096,), "u8"), dq=F((2, 4, 8, 64)), dk=F((2, 2, 8, 64)),
                    dv=F((2, 2, 8, 64)), lse=F((2, 4, 8), "f32"))
    mha.mha.mha_linear_fwd(F((4, 16, 64)), F((64, 32)), F((32,)), out=F((4, 16, 32)), stream=0)
    B, T, S, d, H, Hkv, dk = 2, 16, 24, 128, 2, 1, 64
    sub = dict(mem=F((B, S, d)), H=H, H_kv=Hkv, mask_kind=2, key_lengths=kl, out=F((B, T, d)),
               stream=0)
    ws = [F((B, T, d)), F((d, H * dk)), F((d, Hkv * dk)), F((d, Hkv * dk)), F((H * dk, d))]
    mha.mha.mha_sublayer_fwd(*ws, workspace=F((1 << 20,), "u8"), **sub)
    mha.mha.mha_sublayer_fwd_static(*ws, **sub)
    rec.calls = [c for c in rec.calls if not c[0].endswith("_workspace_size")]
    names = [c[0] for c in rec.calls]
    assert names == ["mha_fwd", "mha_fwd_ex", "mha_bwd", "mha_fwd_lse", "mha_bwd_lse",
                     "mha_linear_fwd", "mha_sublayer_fwd", "mha_sublayer_fwd_static"]
    for name, args in rec.calls:
        assert len(args) == len(getattr(real, name).argtypes), name
    a = dict(rec.calls)
    assert a["mha_fwd"][4:11] == (2, 4, 8, 8, 64, 64, 2)  # B, H, Lq, Lk, d_k, d_v, mask
    assert a["mha_fwd_ex"][4:13] == (2, 4, 2, 8, 8, 64, 64, 0, 2)  # ..., H_kv, ..., layout, mask
    assert a["mha_bwd"][8:17] == (2, 4, 2, 8, 8, 64, 64, 0, 2)
    assert a["mha_bwd"][-2] == 4096  # workspace bytes
    assert a["mha_fwd_lse"][5:14] == (2, 4, 2, 8, 8, 64, 64, 0, 2)  # after out and lse
    assert a["mha_bwd_lse"][9:18] == (2, 4, 2, 8, 8, 64, 64, 0, 2)  # after the gradients
    assert a["mha_linear_fwd"][4:8] == (64, 64, 32, 1)  # M, K, N, dtype
    assert a["mha_sublayer_fwd"][11:19] == (B, T, S, d, H, Hkv, dk, dk)
    assert a["mha_sublayer_fwd"][-2] == 1 << 20
    assert a["mha_sublayer_fwd_static"][11:19] == (B, T, S, d, H, Hkv, dk, dk)
