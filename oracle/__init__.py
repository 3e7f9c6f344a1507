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

MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING, MASK_QUERY_PADDING = 0, 1, 2, 4
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
