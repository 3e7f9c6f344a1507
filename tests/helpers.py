"""Shared helpers for the GPU parity tests: seeded inputs, the CUDA call
through the C ABI binding, the oracle call, and the comparison."""
from __future__ import annotations

import numpy as np

import gen
import oracle

TOL = {"f32": dict(max=1e-4, mean=1e-4), "bf16": dict(max=2e-2, mean=2e-3)}


def to_device(a, dtype, dev="cuda"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype == "bf16":
        t = t.view(torch.bfloat16)
    return t.to(dev)


def from_device(t) -> np.ndarray:
    import torch
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def as_f64(a, dtype):
    return gen.as_f64(a, dtype)


def run_gpu(q, k, v, lens, spec, scale=None, mask=None):
    """The CUDA path on one case: mha_fwd for plain multi-head attention in
    [B, H, L, d], mha_fwd_ex for shared key/value heads or [B, L, H, d]."""
    import torch
    import transformer_head_scaled_mha_gb300 as mha
    dt = spec["dtype"]
    scale = gen.default_scale(spec["dk"]) if scale is None else scale
    mask = spec["mask"] if mask is None else mask
    kl = torch.from_numpy(np.asarray(lens, dtype=np.int32)).cuda() if lens is not None else None
    layout = spec.get("layout", "bhsd")
    args = (to_device(q, dt), to_device(k, dt), to_device(v, dt))
    if layout == "bhsd" and spec.get("Hkv", spec["H"]) == spec["H"]:
        out = mha.mha_fwd(*args, mask_kind=mask, key_lengths=kl, scale=scale)
    else:
        out = mha.mha_fwd_ex(*args, layout=layout, mask_kind=mask, key_lengths=kl, scale=scale)
    torch.cuda.synchronize()
    return from_device(out)


def compare(out_raw, ref, dtype, rows=None, lens=None, spec=None, label=""):
    """Element-wise comparison with the benchmark spec's tolerances.

    out_raw: stored output (uint16 bf16 bits or float32), full [B,H,Lq,dv].
    ref: oracle output, [B,H,Lq,dv] or [len(rows), dv] when ``rows`` is given.
    Returns (max_abs, mean_abs).
    """
    out = as_f64(out_raw, dtype)
    if rows is not None:
        out = out.reshape(-1, out.shape[-1])[rows]
    assert np.isfinite(out).all(), label + ": non-finite output"
    err = np.abs(out - ref)
    tol = TOL[dtype]
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert mx <= tol["max"], "%s: max|err| %.3g > %.3g" % (label, mx, tol["max"])
    assert mean <= tol["mean"], "%s: mean|err| %.3g > %.3g" % (label, mean, tol["mean"])
    # rows the oracle writes as exact zeros must be +0.0 bit for bit
    zero_rows = np.all(ref == 0.0, axis=-1)
    if zero_rows.any():
        raw = out_raw.reshape(-1, out_raw.shape[-1])
        raw = raw[rows] if rows is not None else raw
        zr = zero_rows.reshape(-1)
        assert np.all(raw[zr] == 0), label + ": padded / empty rows are not +0.0"
    return mx, mean


def check_case(spec, seed=0, rows=None, scale=None, mask=None, label=""):
    q, k, v, lens = gen.make_inputs(spec, seed=seed)
    mask = spec["mask"] if mask is None else mask
    scale = gen.default_scale(spec["dk"]) if scale is None else scale
    layout = spec.get("layout", "bhsd")
    out = run_gpu(q, k, v, lens, spec, scale=scale, mask=mask)
    ref = oracle.mha_fwd(q, k, v, mask_kind=mask, key_lengths=lens, scale=scale, rows=rows,
                         layout=layout)
    if layout == "bshd":  # compare in [B, H, L, d], where logical row indices apply
        out = np.ascontiguousarray(out.transpose(0, 2, 1, 3))
        if rows is None:
            ref = np.ascontiguousarray(ref.transpose(0, 2, 1, 3))
    return compare(out, ref, spec["dtype"], rows=rows, label=label or str(spec))


def spec(B, H, Lq, Lk, d, dtype="bf16", mask=0, len_range=None, amp=1.0, Hkv=None,
         layout="bhsd"):
    return dict(B=B, H=H, Lq=Lq, Lk=Lk, dk=d, dv=d, dtype=dtype, amp=amp, mask=mask,
                len_range=len_range, Hkv=H if Hkv is None else Hkv, layout=layout)
