"""Python binding of the C ABI in include/mha.h (ctypes; argument marshalling only).

Every function here forwards to the CUDA library libmha.so built from
``csrc/``.  There is no fallback: if the library is missing or fails to load,
the import raises.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

MHA_DTYPE_F32, MHA_DTYPE_BF16 = 0, 1
MHA_MASK_NONE, MHA_MASK_CAUSAL, MHA_MASK_KEY_PADDING, MHA_MASK_QUERY_PADDING = 0, 1, 2, 4
MHA_MASK_CAUSAL_TAIL = 8
MHA_OK, MHA_ERR_INVALID_ARGUMENT, MHA_ERR_UNSUPPORTED, MHA_ERR_CUDA, MHA_ERR_TIMEOUT = range(5)
PATH_NAMES = {0: "none", 1: "f32_simt", 2: "short_tc", 3: "long_tc", 4: "zero_fill",
              5: "decode_tc"}

MHA_LAYOUT_BHSD, MHA_LAYOUT_BSHD = 0, 1

EXPORTED = ("mha_fwd", "mha_fwd_ex", "mha_fwd_lse", "mha_bwd_lse", "mha_linear_fwd",
            "mha_sublayer_workspace_size",
            "mha_sublayer_fwd", "mha_sublayer_fwd_static", "mha_bwd_workspace_size", "mha_bwd",
            "mha_fwd_path", "mha_fwd_path_ex",
            "mha_status_string", "mha_debug_status", "mha_debug_set_wait", "mha_version")


class MhaError(RuntimeError):
    def __init__(self, status: int, what: str = "mha_fwd"):
        self.status = status
        super().__init__("%s: %s (status %d)" % (what, status_string(status), status))


def _load() -> ctypes.CDLL:
    path = _build.LIB
    if not os.path.exists(path):
        raise ImportError("libmha.so is not built (%s); run __graft_entry__.build() or "
                          "python -m transformer_head_scaled_mha_gb300._build" % path)
    lib = ctypes.CDLL(path)
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    lib.mha_fwd.restype = i32
    lib.mha_fwd.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp,
                            ctypes.c_float, i32, vp]
    lib.mha_fwd_ex.restype = i32
    lib.mha_fwd_ex.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, i32, vp,
                               ctypes.c_float, i32, vp]
    lib.mha_linear_fwd.restype = i32
    lib.mha_fwd_lse.restype = i32
    lib.mha_fwd_lse.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                vp, ctypes.c_float, i32, vp]
    lib.mha_bwd_lse.restype = i32
    lib.mha_bwd_lse.argtypes = [vp] * 9 + [i32] * 9 + [vp, ctypes.c_float, i32, vp,
                                                       ctypes.c_size_t, vp]
    lib.mha_linear_fwd.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp]
    lib.mha_sublayer_workspace_size.restype = ctypes.c_size_t
    lib.mha_sublayer_workspace_size.argtypes = [i32] * 8
    lib.mha_sublayer_fwd.restype = i32
    lib.mha_sublayer_fwd.argtypes = [vp] * 11 + [i32] * 9 + [vp, ctypes.c_float, i32, vp,
                                                            ctypes.c_size_t, vp]
    lib.mha_sublayer_fwd_static.restype = i32
    lib.mha_sublayer_fwd_static.argtypes = [vp] * 11 + [i32] * 9 + [vp, ctypes.c_float, i32, vp]
    lib.mha_bwd_workspace_size.restype = ctypes.c_size_t
    lib.mha_bwd_workspace_size.argtypes = [i32] * 3
    lib.mha_bwd.restype = i32
    lib.mha_bwd.argtypes = [vp] * 8 + [i32] * 9 + [vp, ctypes.c_float, i32, vp, ctypes.c_size_t,
                                                    vp]
    lib.mha_fwd_path.restype = i32
    lib.mha_fwd_path.argtypes = [i32] * 8
    lib.mha_fwd_path_ex.restype = i32
    lib.mha_fwd_path_ex.argtypes = [i32] * 9
    lib.mha_status_string.restype = ctypes.c_char_p
    lib.mha_status_string.argtypes = [i32]
    lib.mha_debug_status.restype = i32
    lib.mha_debug_status.argtypes = [vp]
    lib.mha_debug_set_wait.restype = i32
    lib.mha_debug_set_wait.argtypes = [ctypes.c_ulonglong, i32]
    lib.mha_version.restype = i32
    lib.mha_version.argtypes = []
    return lib


lib = _load()
LIB_PATH = _build.LIB


def status_string(status: int) -> str:
    return lib.mha_status_string(int(status)).decode()


mha_status_string = status_string


def mha_version() -> int:
    return int(lib.mha_version())


def mha_fwd_path(B, H, Lq, Lk, d_k, d_v, mask_kind, dtype) -> int:
    return int(lib.mha_fwd_path(B, H, Lq, Lk, d_k, d_v, mask_kind, dtype))


def mha_fwd_path_ex(B, H, H_kv, Lq, Lk, d_k, d_v, mask_kind, dtype) -> int:
    return int(lib.mha_fwd_path_ex(B, H, H_kv, Lq, Lk, d_k, d_v, mask_kind, dtype))


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def mha_debug_status(stream=None) -> int:
    return int(lib.mha_debug_status(_stream_handle(stream)))


def mha_debug_set_wait(limit_ns: int = 0, stall: int = 0) -> int:
    """Test hook: the kernels' wait limit in ns (0: the default 2 s) and the
    stall bits that make a kernel wait on a barrier nothing signals."""
    return int(lib.mha_debug_set_wait(int(limit_ns), int(stall)))


def _lengths_ptr(key_lengths, B, device):
    """Device address of the per-sequence lengths (None when not given)."""
    import torch
    if key_lengths is None:
        return None
    if key_lengths.dtype != torch.int32 or not key_lengths.is_cuda or \
            key_lengths.numel() != B or not key_lengths.is_contiguous() or \
            key_lengths.device != device:
        raise ValueError("key_lengths must be a contiguous int32 CUDA tensor of shape [B] on "
                         "the inputs' device")
    return key_lengths.data_ptr()


def _workspace_bytes(workspace, device):
    """Size in bytes of a caller's workspace tensor, after checking where it lives."""
    if not workspace.is_cuda or not workspace.is_contiguous() or workspace.device != device:
        raise ValueError("workspace must be a contiguous CUDA tensor on the inputs' device")
    return workspace.numel() * workspace.element_size()


def _marshal(q, k, v, out, key_lengths, scale, layout):
    """Check shapes/dtypes, allocate ``out`` if needed; returns the C arguments."""
    import torch
    if layout not in ("bhsd", "bshd"):
        raise ValueError("layout must be 'bhsd' or 'bshd'")
    if layout == "bshd":
        B, Lq, H, dk = q.shape
        Lk, Hkv, dv = k.shape[1], k.shape[2], v.shape[3]
        kshape, vshape, oshape = (B, Lk, Hkv, dk), (B, Lk, Hkv, dv), (B, Lq, H, dv)
    else:
        B, H, Lq, dk = q.shape
        Hkv, Lk, dv = k.shape[1], k.shape[2], v.shape[3]
        kshape, vshape, oshape = (B, Hkv, Lk, dk), (B, Hkv, Lk, dv), (B, H, Lq, dv)
    if q.dtype == torch.float32:
        dtype = MHA_DTYPE_F32
    elif q.dtype == torch.bfloat16:
        dtype = MHA_DTYPE_BF16
    else:
        raise TypeError("q must be float32 or bfloat16")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype")
    if tuple(k.shape) != kshape or tuple(v.shape) != vshape:
        raise ValueError("shape mismatch: q %s k %s v %s" % (tuple(q.shape), tuple(k.shape),
                                                             tuple(v.shape)))
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA tensor" % name)
        if t.device != q.device:
            raise ValueError("%s must be on q's device" % name)
    if out is None:
        out = torch.empty(oshape, dtype=q.dtype, device=q.device)
    elif tuple(out.shape) != oshape or out.dtype != q.dtype or not out.is_contiguous() or \
            out.device != q.device:
        raise ValueError("out must be a contiguous %s tensor of q's dtype on q's device"
                         % (oshape,))
    kl_ptr = _lengths_ptr(key_lengths, B, q.device)
    if scale is None:
        scale = float(dk) ** -0.5
    return out, (B, H, Hkv, Lq, Lk, dk, dv), kl_ptr, float(scale), dtype


def mha_fwd(q, k, v, out=None, *, mask_kind: int = 0, key_lengths=None, scale=None,
            stream=None):
    """out = softmax(q k^T * scale) v per (batch, head), on q's CUDA device.

    q [B,H,Lq,d_k], k [B,H,Lk,d_k], v [B,H,Lk,d_v]: contiguous CUDA tensors, all
    float32 or all bfloat16.  ``key_lengths``: int32 CUDA tensor [B] (needed for
    the padding masks).  ``scale`` defaults to 1/sqrt(d_k).  Enqueued on
    ``stream`` (default: torch's current stream); returns ``out``.
    """
    import torch
    out, (B, H, Hkv, Lq, Lk, dk, dv), kl_ptr, scale, dtype = _marshal(q, k, v, out, key_lengths,
                                                                      scale, "bhsd")
    if Hkv != H:
        raise ValueError("mha_fwd needs as many key/value heads as query heads; "
                         "use mha_fwd_ex for shared key/value heads")
    with torch.cuda.device(q.device):
        st = lib.mha_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, Lq, Lk,
                         dk, dv, int(mask_kind), kl_ptr, scale, dtype, _stream_handle(stream))
    if st != MHA_OK:
        raise MhaError(st)
    return out


def mha_fwd_ex(q, k, v, out=None, *, layout: str = "bhsd", mask_kind: int = 0,
               key_lengths=None, scale=None, stream=None):
    """mha_fwd with shared key/value heads and a choice of layout.

    layout "bhsd": q [B,H,Lq,d_k], k [B,H_kv,Lk,d_k], v [B,H_kv,Lk,d_v];
    layout "bshd": q [B,Lq,H,d_k], k [B,Lk,H_kv,d_k], v [B,Lk,H_kv,d_v]; ``out``
    has q's layout.  H_kv (from k) divides H; query head h reads key/value head
    h // (H // H_kv).
    """
    import torch
    out, (B, H, Hkv, Lq, Lk, dk, dv), kl_ptr, scale, dtype = _marshal(q, k, v, out, key_lengths,
                                                                      scale, layout)
    with torch.cuda.device(q.device):
        st = lib.mha_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, Hkv,
                            Lq, Lk, dk, dv, MHA_LAYOUT_BSHD if layout == "bshd" else
                            MHA_LAYOUT_BHSD, int(mask_kind), kl_ptr, scale, dtype,
                            _stream_handle(stream))
    if st != MHA_OK:
        raise MhaError(st, "mha_fwd_ex")
    return out


def _lse_tensor(lse, B, H, Lq, device):
    import torch
    if lse is None:
        return torch.empty((B, H, Lq), dtype=torch.float32, device=device)
    if tuple(lse.shape) != (B, H, Lq) or lse.dtype != torch.float32 or not lse.is_contiguous() \
            or lse.device != device:
        raise ValueError("lse must be a contiguous float32 tensor of shape %s on q's device"
                         % ((B, H, Lq),))
    return lse


def mha_fwd_lse(q, k, v, out=None, lse=None, *, layout: str = "bhsd", mask_kind: int = 0,
                key_lengths=None, scale=None, stream=None):
    """mha_fwd_ex that also returns each row's softmax statistics ``lse``
    [B, H, Lq] (float32, base 2, +inf for rows stored as zeros), which
    mha_bwd_lse takes.  Returns (out, lse)."""
    import torch
    out, (B, H, Hkv, Lq, Lk, dk, dv), kl_ptr, scale, dtype = _marshal(q, k, v, out, key_lengths,
                                                                      scale, layout)
    lse = _lse_tensor(lse, B, H, Lq, q.device)
    with torch.cuda.device(q.device):
        st = lib.mha_fwd_lse(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                             lse.data_ptr(), B, H, Hkv, Lq, Lk, dk, dv,
                             MHA_LAYOUT_BSHD if layout == "bshd" else MHA_LAYOUT_BHSD,
                             int(mask_kind), kl_ptr, scale, dtype, _stream_handle(stream))
    if st != MHA_OK:
        raise MhaError(st, "mha_fwd_lse")
    return out, lse


def mha_bwd_workspace_size(B, H, Lq) -> int:
    return int(lib.mha_bwd_workspace_size(B, H, Lq))


def mha_bwd(q, k, v, out, dout, *, layout: str = "bhsd", mask_kind: int = 0, key_lengths=None,
            scale=None, workspace=None, dq=None, dk=None, dv=None, stream=None, lse=None):
    """Gradients (dq, dk, dv) of a loss through mha_fwd_ex, given its output
    ``out`` and the incoming gradient ``dout`` (out's shape).  Same layouts,
    shared key/value heads, masks and scale as mha_fwd_ex.  ``workspace``: a
    uint8 CUDA tensor of at least mha_bwd_workspace_size(B, H, Lq) bytes, or
    None to allocate one.  ``lse``: the forward's row statistics from
    mha_fwd_lse (then mha_bwd_lse runs: no statistics pass), or None."""
    import torch
    _, (B, H, Hkv, Lq, Lk, dk_, dv_), kl_ptr, scale, dtype = _marshal(q, k, v, out, key_lengths,
                                                                      scale, layout)
    if dout.shape != out.shape or dout.dtype != q.dtype or not dout.is_contiguous() or \
            dout.device != q.device:
        raise ValueError("dout must be a contiguous tensor like out")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, g, ref in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        if g.shape != ref.shape or g.dtype != ref.dtype or not g.is_contiguous() or \
                g.device != ref.device:
            raise ValueError("%s must be a contiguous tensor like its input" % name)
    n = mha_bwd_workspace_size(B, H, Lq)
    if workspace is None:
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=q.device)
    ws_bytes = _workspace_bytes(workspace, q.device)
    lay = MHA_LAYOUT_BSHD if layout == "bshd" else MHA_LAYOUT_BHSD
    with torch.cuda.device(q.device):
        if lse is None:
            st = lib.mha_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                             dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H,
                             Hkv, Lq, Lk, dk_, dv_, lay, int(mask_kind), kl_ptr, scale, dtype,
                             workspace.data_ptr(), ws_bytes, _stream_handle(stream))
        else:
            lse = _lse_tensor(lse, B, H, Lq, q.device)
            st = lib.mha_bwd_lse(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                 dout.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                 dv.data_ptr(), B, H, Hkv, Lq, Lk, dk_, dv_, lay, int(mask_kind),
                                 kl_ptr, scale, dtype, workspace.data_ptr(), ws_bytes,
                                 _stream_handle(stream))
    if st != MHA_OK:
        raise MhaError(st, "mha_bwd" if lse is None else "mha_bwd_lse")
    return dq, dk, dv


def _bf16_cuda(name, t, ndim=None):
    import torch
    if t is None:
        return None
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError("%s must be a contiguous bfloat16 CUDA tensor" % name)
    if ndim is not None and t.dim() != ndim:
        raise ValueError("%s must have %d dimensions" % (name, ndim))
    return t


def mha_linear_fwd(x, w, b=None, out=None, *, stream=None):
    """y = x W + b: x [..., K], W [K, N] (input-major), b [N] or None; bfloat16."""
    import torch
    _bf16_cuda("x", x)
    _bf16_cuda("w", w, 2)
    _bf16_cuda("b", b, 1)
    K, N = w.shape
    if x.shape[-1] != K or (b is not None and b.shape[0] != N):
        raise ValueError("shape mismatch: x %s w %s" % (tuple(x.shape), tuple(w.shape)))
    for name, t in (("w", w), ("b", b), ("out", out)):
        if t is not None and t.device != x.device:
            raise ValueError("%s must be on x's device" % name)
    M = x.numel() // K if K else 0
    if out is None:
        out = torch.empty(tuple(x.shape[:-1]) + (N,), dtype=x.dtype, device=x.device)
    else:
        _bf16_cuda("out", out)
        if tuple(out.shape) != tuple(x.shape[:-1]) + (N,):
            raise ValueError("out must have shape %s" % ((tuple(x.shape[:-1]) + (N,)),))
    with torch.cuda.device(x.device):
        st = lib.mha_linear_fwd(x.data_ptr(), w.data_ptr(), b.data_ptr() if b is not None else None,
                                out.data_ptr(), M, K, N, MHA_DTYPE_BF16, _stream_handle(stream))
    if st != MHA_OK:
        raise MhaError(st, "mha_linear_fwd")
    return out


def mha_sublayer_workspace_size(B, T, S, d_model, H, H_kv, d_k, d_v) -> int:
    return int(lib.mha_sublayer_workspace_size(B, T, S, d_model, H, H_kv, d_k, d_v))


def _sublayer_marshal(x, w_q, w_k, w_v, w_o, b_q, b_k, b_v, b_o, mem, H, H_kv, key_lengths,
                      scale, out):
    """Check the sublayer's tensors against one another (shapes, dtype, device);
    returns (out, (B, T, S, d_model, H, H_kv, d_k, d_v), lengths pointer, scale,
    memory pointer).  The library sizes every buffer from these dimensions, so
    a tensor that disagrees with them is refused here."""
    import torch
    H_kv = H if H_kv is None else H_kv
    _bf16_cuda("x", x, 3)
    _bf16_cuda("mem", mem, 3)
    for name, t in (("w_q", w_q), ("w_k", w_k), ("w_v", w_v), ("w_o", w_o)):
        _bf16_cuda(name, t, 2)
    for name, t in (("b_q", b_q), ("b_k", b_k), ("b_v", b_v), ("b_o", b_o)):
        _bf16_cuda(name, t, 1)
    B, T, d_model = x.shape
    S = mem.shape[1] if mem is not None else T
    if H <= 0 or H_kv <= 0 or w_q.shape[1] % H or w_v.shape[1] % H_kv:
        raise ValueError("the projection widths must be whole multiples of the head counts")
    d_k, d_v = w_q.shape[1] // H, w_v.shape[1] // H_kv
    want = {"w_q": (w_q, (d_model, H * d_k)), "w_k": (w_k, (d_model, H_kv * d_k)),
            "w_v": (w_v, (d_model, H_kv * d_v)), "w_o": (w_o, (H * d_v, d_model)),
            "b_q": (b_q, (H * d_k,)), "b_k": (b_k, (H_kv * d_k,)), "b_v": (b_v, (H_kv * d_v,)),
            "b_o": (b_o, (d_model,)), "mem": (mem, (B, S, d_model))}
    for name, (t, shape) in want.items():
        if t is None:
            continue
        if tuple(t.shape) != shape:
            raise ValueError("%s must have shape %s, not %s" % (name, shape, tuple(t.shape)))
        if t.device != x.device:
            raise ValueError("%s must be on x's device" % name)
    if out is None:
        out = torch.empty((B, T, d_model), dtype=x.dtype, device=x.device)
    else:
        _bf16_cuda("out", out, 3)
        if tuple(out.shape) != (B, T, d_model) or out.device != x.device:
            raise ValueError("out must have shape %s on x's device" % ((B, T, d_model),))
    kl_ptr = _lengths_ptr(key_lengths, B, x.device)
    if scale is None:
        scale = float(d_k) ** -0.5
    # an empty memory (S = 0) is never read; pass a non-null stand-in so it is
    # not taken for self-attention
    mem_ptr = None if mem is None else (mem.data_ptr() if mem.numel() else x.data_ptr())
    return out, (B, T, S, d_model, H, H_kv, d_k, d_v), kl_ptr, float(scale), mem_ptr


def mha_sublayer_fwd(x, w_q, w_k, w_v, w_o, b_q=None, b_k=None, b_v=None, b_o=None, *, mem=None,
                     H, H_kv=None, mask_kind: int = 0, key_lengths=None, scale=None,
                     workspace=None, out=None, stream=None):
    """Multi-head attention sublayer (projections, attention, output projection).

    x [B, T, d_model]; mem [B, S, d_model] or None (self-attention); weights
    input-major: W_q [d_model, H d_k], W_k/W_v [d_model, H_kv d], W_o [H d_v,
    d_model]; biases optional.  ``workspace``: a uint8 CUDA tensor of at least
    mha_sublayer_workspace_size(...) bytes (allocated here when None).
    """
    import torch
    out, dims, kl_ptr, scale, mem_ptr = _sublayer_marshal(
        x, w_q, w_k, w_v, w_o, b_q, b_k, b_v, b_o, mem, H, H_kv, key_lengths, scale, out)
    if workspace is None:
        workspace = torch.empty(max(mha_sublayer_workspace_size(*dims), 1), dtype=torch.uint8,
                                device=x.device)
    ws_bytes = _workspace_bytes(workspace, x.device)
    ptr = lambda t: t.data_ptr() if t is not None else None
    with torch.cuda.device(x.device):
        st = lib.mha_sublayer_fwd(ptr(x), mem_ptr, ptr(out), ptr(w_q), ptr(w_k), ptr(w_v),
                                  ptr(w_o), ptr(b_q), ptr(b_k), ptr(b_v), ptr(b_o), *dims,
                                  int(mask_kind), kl_ptr, scale, MHA_DTYPE_BF16,
                                  workspace.data_ptr(), ws_bytes, _stream_handle(stream))
    if st != MHA_OK:
        raise MhaError(st, "mha_sublayer_fwd")
    return out


def mha_sublayer_fwd_static(x, w_q, w_k, w_v, w_o, b_q=None, b_k=None, b_v=None, b_o=None, *,
                            mem=None, H, H_kv=None, mask_kind: int = 0, key_lengths=None,
                            scale=None, out=None, stream=None):
    """mha_sublayer_fwd on the library's static device scratch (no workspace,
    nothing allocated per call; calls that overlap in time race on the
    scratch).  Raises MhaError (unsupported) above 64 MiB of intermediates."""
    import torch
    out, dims, kl_ptr, scale, mem_ptr = _sublayer_marshal(
        x, w_q, w_k, w_v, w_o, b_q, b_k, b_v, b_o, mem, H, H_kv, key_lengths, scale, out)
    ptr = lambda t: t.data_ptr() if t is not None else None
    with torch.cuda.device(x.device):
        st = lib.mha_sublayer_fwd_static(ptr(x), mem_ptr, ptr(out), ptr(w_q), ptr(w_k),
                                         ptr(w_v), ptr(w_o), ptr(b_q), ptr(b_k), ptr(b_v),
                                         ptr(b_o), *dims, int(mask_kind), kl_ptr, scale,
                                         MHA_DTYPE_BF16, _stream_handle(stream))
    if st != MHA_OK:
        raise MhaError(st, "mha_sublayer_fwd_static")
    return out
