"""fp64 CPU oracle for multi-head scaled dot-product attention.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg use it to check and time the CUDA path.  The product
package never imports it.  It shares no code with the CUDA path; the only
module both sides use is ``gen`` (seeded inputs, no attention arithmetic).

The arithmetic lives in ``mha_oracle.c`` (plain C, IEEE double, row by row;
see its header for the steps and the passages they follow).  This wrapper
compiles it with gcc and marshals numpy arrays.

Every function here is pinned by ``tests/test_oracle.py`` against values the
pages print (the three-token worked example), closed forms, invariants and a
50-digit brute force.

``mha_bwd`` is the backward pass: the gradients of a loss through the
attention, by the chain rule through the same steps (for training, as the
pages describe it; ``mha_oracle.c`` states the formulas).

``linear`` and ``mha_sublayer`` add the steps on either side of the attention:
the learned projections with their biases, the head split and concatenation,
and the output projection (trishampatil.com, "Multi-Head Attention" and "The
Output Projection W^O"; aicassindra.com, "A faithful layer in code").  The
matrix products there are numpy float64 matmuls (a library primitive used as
one step); the attention step is the C oracle above.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mha_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libmha_oracle.so")

MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING, MASK_QUERY_PADDING, MASK_CAUSAL_TAIL = 0, 1, 2, 4, 8
_IN_CODES = {np.dtype(np.float64): 0, np.dtype(np.float32): 1, np.dtype(np.uint16): 2}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no FP contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.oracle_mha_rows_ex_f64.restype = ctypes.c_int
            lib.oracle_mha_rows_ex_f64.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_void_p, ctypes.c_double,
                ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.oracle_mha_bwd_f64.restype = ctypes.c_int
            lib.oracle_mha_bwd_f64.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_void_p, ctypes.c_double,
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def mha_fwd(q, k, v, *, mask_kind: int = 0, key_lengths=None, scale: float,
            rows=None, threads: int = 0, return_weights: bool = False,
            return_scores: bool = False, layout: str = "bhsd"):
    """Attention output in float64.

    layout "bhsd": q [B,H,Lq,dk], k [B,Hkv,Lk,dk], v [B,Hkv,Lk,dv];
    layout "bshd": q [B,Lq,H,dk], k [B,Lk,Hkv,dk], v [B,Lk,Hkv,dv].
    Hkv (taken from k) divides H; query head h reads key/value head
    h // (H // Hkv).  Arrays: float64, float32 or uint16 (bfloat16 bit
    patterns), all the same type.  ``key_lengths`` int [B].
    ``rows``: optional logical row indices (b*H + h)*Lq + i; then the result is
    [len(rows), dv] (and [len(rows), Lk] for weights/scores), else the output
    in the inputs' layout and weights/scores as [B,H,Lq,Lk].
    """
    q = np.ascontiguousarray(q)
    k = np.ascontiguousarray(k)
    v = np.ascontiguousarray(v)
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in _IN_CODES:
        raise TypeError("q, k, v must share one of float64, float32, uint16(bf16)")
    if layout not in ("bhsd", "bshd"):
        raise ValueError("layout must be 'bhsd' or 'bshd'")
    bshd = layout == "bshd"
    if bshd:
        B, Lq, H, dk = q.shape
        Bk, Lk, Hkv, dk2 = k.shape
        Bv, Lk2, Hv, dv = v.shape
    else:
        B, H, Lq, dk = q.shape
        Bk, Hkv, Lk, dk2 = k.shape
        Bv, Hv, Lk2, dv = v.shape
    if (Bk, dk2) != (B, dk) or (Bv, Hv, Lk2) != (B, Hkv, Lk):
        raise ValueError("shape mismatch")
    if Hkv <= 0 and H > 0 or (Hkv > 0 and H % Hkv):
        raise ValueError("key/value heads must divide query heads")
    kl = None
    if key_lengths is not None:
        kl = np.ascontiguousarray(key_lengths, dtype=np.int32)
        if kl.shape != (B,):
            raise ValueError("key_lengths must have shape [B]")
    if rows is None:
        rows_a = None
        nrows = B * H * Lq
        oshape, wshape = (B, H, Lq, dv), (B, H, Lq, Lk)
    else:
        rows_a = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = rows_a.shape[0]
        oshape, wshape = (nrows, dv), (nrows, Lk)
    out = np.zeros(oshape, dtype=np.float64)
    w = np.zeros(wshape, dtype=np.float64) if return_weights else None
    s = np.zeros(wshape, dtype=np.float64) if return_scores else None
    rc = _load().oracle_mha_rows_ex_f64(
        _ptr(q), _ptr(k), _ptr(v), _IN_CODES[q.dtype], B, H, max(Hkv, 1) if H == 0 else Hkv,
        Lq, Lk, dk, dv, 1 if bshd else 0,
        int(mask_kind), _ptr(kl), float(scale), _ptr(rows_a), nrows,
        _ptr(out), _ptr(w), _ptr(s), int(threads))
    if rc != 0:
        raise ValueError("oracle rejected the arguments (rc=%d)" % rc)
    if rows is None and bshd:
        out = np.ascontiguousarray(out.transpose(0, 2, 1, 3))
    res = [out]
    if return_weights:
        res.append(w)
    if return_scores:
        res.append(s)
    return res[0] if len(res) == 1 else tuple(res)


def mha_bwd(q, k, v, dout, *, mask_kind: int = 0, key_lengths=None, scale: float,
            layout: str = "bhsd", units=None, rows=None, threads: int = 0):
    """Gradients (dq, dk, dv) in float64 of L = sum(out * dout) through ``mha_fwd``.

    Same shapes, layouts, dtypes and masks as ``mha_fwd``; ``dout`` has the
    output's shape and the inputs' dtype.  The steps are the chain rule through
    the forward (see ``mha_oracle.c``).  ``units``: optional logical (batch
    element, key/value head) indices b * Hkv + g to compute (others stay 0);
    ``rows``: optional (lo, hi) range of query rows taken in each unit (a
    timing sample; gradients are then partial sums).
    """
    q, k, v, dout = (np.ascontiguousarray(a) for a in (q, k, v, dout))
    if not (q.dtype == k.dtype == v.dtype == dout.dtype) or q.dtype not in _IN_CODES:
        raise TypeError("q, k, v, dout must share one of float64, float32, uint16(bf16)")
    if layout not in ("bhsd", "bshd"):
        raise ValueError("layout must be 'bhsd' or 'bshd'")
    bshd = layout == "bshd"
    if bshd:
        B, Lq, H, dk = q.shape
        Bk, Lk, Hkv, dk2 = k.shape
        Bv, Lk2, Hv, dv = v.shape
        oshape = (B, Lq, H, dv)
    else:
        B, H, Lq, dk = q.shape
        Bk, Hkv, Lk, dk2 = k.shape
        Bv, Hv, Lk2, dv = v.shape
        oshape = (B, H, Lq, dv)
    if (Bk, dk2) != (B, dk) or (Bv, Hv, Lk2) != (B, Hkv, Lk) or dout.shape != oshape:
        raise ValueError("shape mismatch")
    if Hkv <= 0 and H > 0 or (Hkv > 0 and H % Hkv):
        raise ValueError("key/value heads must divide query heads")
    kl = None
    if key_lengths is not None:
        kl = np.ascontiguousarray(key_lengths, dtype=np.int32)
        if kl.shape != (B,):
            raise ValueError("key_lengths must have shape [B]")
    units_a = None if units is None else np.ascontiguousarray(units, dtype=np.int64)
    nunits = B * Hkv if units_a is None else units_a.shape[0]
    i_lo, i_hi = (0, Lq) if rows is None else (int(rows[0]), int(rows[1]))
    dq = np.zeros(q.shape, dtype=np.float64)
    dkk = np.zeros(k.shape, dtype=np.float64)
    dvv = np.zeros(v.shape, dtype=np.float64)
    rc = _load().oracle_mha_bwd_f64(
        _ptr(q), _ptr(k), _ptr(v), _ptr(dout), _IN_CODES[q.dtype], B, H,
        max(Hkv, 1) if H == 0 else Hkv, Lq, Lk, dk, dv, 1 if bshd else 0, int(mask_kind),
        _ptr(kl), float(scale), _ptr(units_a), nunits, i_lo, i_hi, _ptr(dq), _ptr(dkk), _ptr(dvv),
        int(threads))
    if rc != 0:
        raise ValueError("oracle rejected the arguments (rc=%d)" % rc)
    return dq, dkk, dvv


def _f64(a):
    """Stored values (float64, float32, or uint16 bfloat16 bits) widened exactly."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def linear(x, w, b=None):
    """y = x W + b in float64.

    x [..., d_in], W [d_in, d_out], b [d_out] (or None): the learned projection
    of a token vector, written input-major as in "Q · W_i^Q" with
    W_i^Q of shape d_model x d_k; the bias is the one every linear layer of the
    faithful layer carries.  Inputs may be float64, float32 or bfloat16 bits.
    """
    y = _f64(x) @ _f64(w)
    if b is not None:
        y = y + _f64(b)
    return y


def mha_sublayer(x, mem, w_q, w_k, w_v, w_o, b_q=None, b_k=None, b_v=None, b_o=None, *,
                 H: int, H_kv: int = None, mask_kind: int = 0, key_lengths=None, scale=None):
    """Multi-head attention sublayer in float64.

    x [B, T, d_model] (queries), mem [B, S, d_model] (keys and values; pass x
    for self-attention); W_q [d_model, H d_k], W_k and W_v [d_model, H_kv d_k],
    W_o [H d_v, d_model]; biases of the output widths (or None).
      1. q = x W_q + b_q, k = mem W_k + b_k, v = mem W_v + b_v
      2. head i of q is columns [i d_k, (i + 1) d_k) (same for k, v), i.e. the
         projections viewed as [B, L, heads, d]
      3. head_i = Attention(q_i, k_g, v_g), g = i / (H / H_kv)  (the C oracle)
      4. concatenate the heads back to [B, T, H d_v] and project:
         out = concat W_o + b_o
    ``scale`` defaults to 1/sqrt(d_k).  Returns float64 [B, T, d_out].
    """
    H_kv = H if H_kv is None else H_kv
    q = linear(x, w_q, b_q)
    k = linear(mem, w_k, b_k)
    v = linear(mem, w_v, b_v)
    B, T, hq = q.shape
    S = k.shape[1]
    if hq % H or k.shape[2] % H_kv or v.shape[2] % H_kv:
        raise ValueError("projection widths must split into heads")
    dk, dv = hq // H, v.shape[2] // H_kv
    if k.shape[2] // H_kv != dk:
        raise ValueError("query and key head widths differ")
    if scale is None:
        scale = 1.0 / np.sqrt(dk)
    heads = mha_fwd(q.reshape(B, T, H, dk), k.reshape(B, S, H_kv, dk),
                    v.reshape(B, S, H_kv, dv), mask_kind=mask_kind, key_lengths=key_lengths,
                    scale=scale, layout="bshd")
    return linear(heads.reshape(B, T, H * dv), w_o, b_o)
