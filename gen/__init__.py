"""Seeded synthetic inputs for multi-head scaled dot-product attention.

This module is the only code shared by the CPU oracle, the tests and the
bench.  It draws numbers and rounds them to a storage format; it holds none of
the attention arithmetic.

Random numbers
--------------
SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014) used as a counter-based generator: the n-th 64-bit
word of stream ``s`` under seed ``seed`` is ``mix64(key + (n + 1) * GAMMA)``
with ``key = mix64(seed * GAMMA ^ (s + 1) * STREAM_MUL)``.  ``mix64`` is the
SplitMix64 output finaliser.  Each tensor gets its own stream (Q=0, K=1, V=2,
key lengths=3), so tensors can be drawn independently and in any order.

Normal variates: uniforms in (0, 1) from the top 53 bits, ``u = (w >> 11 +
0.5) * 2**-53``; Box-Muller on consecutive pairs (u1, u2): element 2m gets
``sqrt(-2 ln u1) cos(2 pi u2)`` and element 2m+1 gets the matching sine.  The
fp64 normal is multiplied by the amplitude and rounded ONCE to the storage type
(round to nearest even): float32 through numpy, bfloat16 by rounding the
float64 bit pattern directly to 8 significant bits.

Lengths: an inclusive integer range [lo, hi] drawn from the top 32 bits of
successive words, rejecting words at or above the largest multiple of the
range size (no modulo bias).

bfloat16 values are kept as their uint16 bit patterns (numpy has no bfloat16).
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
STREAM_MUL = np.uint64(0xD1B54A32D192ED03)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

STREAM_Q, STREAM_K, STREAM_V, STREAM_LENGTHS = 0, 1, 2, 3

_CHUNK = 1 << 22  # elements per vectorised block (bounds host memory)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.array([seed], dtype=np.uint64) * GAMMA
        s ^= np.array([stream + 1], dtype=np.uint64) * STREAM_MUL
        return _mix64(s)[0]


def words(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Counter-based SplitMix64 words ``start .. start+count-1`` of a stream."""
    key = stream_key(seed, stream)
    with np.errstate(over="ignore"):
        n = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        return _mix64(key + n * GAMMA)


def normals_f64(seed: int, stream: int, count: int, start: int = 0) -> np.ndarray:
    """``count`` N(0,1) draws in float64 (Box-Muller over word pairs)."""
    if count == 0:
        return np.zeros(0, dtype=np.float64)
    p0 = start // 2
    p1 = (start + count + 1) // 2
    w = words(seed, stream, 2 * p0, 2 * (p1 - p0))
    u = ((w >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * np.pi * u2
    z = np.empty(2 * (p1 - p0), dtype=np.float64)
    z[0::2] = r * np.cos(t)
    z[1::2] = r * np.sin(t)
    off = start - 2 * p0
    return z[off:off + count]


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 to bfloat16 (nearest, ties to even) in one step.

    Values here are finite and far from the bfloat16 subnormal/overflow range;
    zero maps to +0 or -0 by sign.
    """
    b = np.ascontiguousarray(x, dtype=np.float64).view(np.uint64)
    keep = np.uint64(45)  # 52 - 7 explicit significand bits kept
    lsb = (b >> keep) & np.uint64(1)
    with np.errstate(over="ignore"):
        r = (b + (np.uint64((1 << 44) - 1) + lsb)) & ~np.uint64((1 << 45) - 1)
    f32 = r.view(np.float64).astype(np.float32)  # exact: 8-bit significand
    return (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def tensor(seed: int, stream: int, shape, dtype: str, amp: float = 1.0) -> np.ndarray:
    """N(0,1)*amp tensor of ``shape`` rounded to ``dtype`` ('f32', 'bf16', 'f64').

    'bf16' returns uint16 bit patterns.  Element order is row-major over
    ``shape``; element e consumes normal number e of the stream.
    """
    n = int(np.prod(shape)) if len(shape) else 1
    out_dt = {"f32": np.float32, "bf16": np.uint16, "f64": np.float64}[dtype]
    out = np.empty(n, dtype=out_dt)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        z = normals_f64(seed, stream, c, start=s)
        if amp != 1.0:
            z = z * amp
        if dtype == "f32":
            out[s:s + c] = z.astype(np.float32)
        elif dtype == "bf16":
            out[s:s + c] = f64_to_bf16_bits(z)
        else:
            out[s:s + c] = z
    return out.reshape(shape)


def lengths(seed: int, count: int, lo: int, hi: int, stream: int = STREAM_LENGTHS) -> np.ndarray:
    """``count`` i.i.d. integers uniform on the inclusive range [lo, hi]."""
    if not (0 <= lo <= hi):
        raise ValueError("need 0 <= lo <= hi")
    r = hi - lo + 1
    limit = ((1 << 32) // r) * r
    out = np.empty(count, dtype=np.int32)
    pos = 0
    got = 0
    while got < count:
        w = words(seed, stream, pos, 64)
        pos += 64
        for x in (w >> np.uint64(32)).tolist():
            if x < limit:
                out[got] = lo + x % r
                got += 1
                if got == count:
                    break
    return out


# ---------------------------------------------------------------------------
# Workloads (shapes, value distributions and masks of the five attention
# settings: Transformer-base/big sentence lengths and one long causal context).
# ---------------------------------------------------------------------------
MASK_NONE, MASK_CAUSAL, MASK_KEY_PADDING, MASK_QUERY_PADDING, MASK_CAUSAL_TAIL = 0, 1, 2, 4, 8

WORKLOADS = {
    # fp32 encoder self-attention, no mask
    "enc_f32_b2_h8_l32_d64": dict(B=2, H=8, Lq=32, Lk=32, dk=64, dv=64, dtype="f32",
                                  amp=1.0, mask=MASK_NONE, len_range=None),
    # Transformer-base encoder self-attention with key (and query) padding
    "enc_pad_bf16_b256_h8_l64_d64": dict(B=256, H=8, Lq=64, Lk=64, dk=64, dv=64, dtype="bf16",
                                         amp=1.0, mask=MASK_KEY_PADDING | MASK_QUERY_PADDING,
                                         len_range=(8, 64)),
    # Transformer-base decoder causal self-attention
    "dec_causal_bf16_b128_h8_l128_d64": dict(B=128, H=8, Lq=128, Lk=128, dk=64, dv=64,
                                             dtype="bf16", amp=1.0, mask=MASK_CAUSAL,
                                             len_range=None),
    # Transformer-big encoder-decoder cross-attention, source key padding
    "cross_pad_bf16_b64_h16_lq96_lk128_d64": dict(B=64, H=16, Lq=96, Lk=128, dk=64, dv=64,
                                                  dtype="bf16", amp=1.0, mask=MASK_KEY_PADDING,
                                                  len_range=(16, 128)),
    # long-context causal self-attention, d=128
    "long_causal_bf16_b4_h16_l8192_d128": dict(B=4, H=16, Lq=8192, Lk=8192, dk=128, dv=128,
                                               dtype="bf16", amp=0.5, mask=MASK_CAUSAL,
                                               len_range=None),
    # one generation step of the Transformer-base decoder: one new token per
    # sequence against its cached keys/values (cache lengths U{128..1024})
    "decode_bf16_b256_h8_lk1024_d64": dict(B=256, H=8, Lq=1, Lk=1024, dk=64, dv=64,
                                           dtype="bf16", amp=1.0,
                                           mask=MASK_CAUSAL_TAIL | MASK_KEY_PADDING,
                                           len_range=(128, 1024), layout="bshd"),
    # a generation step with grouped key/value heads and long caches
    # (32 query heads over 8 key/value heads, d=128, lengths U{4096..8192})
    "decode_gqa_bf16_b64_h32_kv8_lk8192_d128": dict(B=64, H=32, Hkv=8, Lq=1, Lk=8192, dk=128,
                                                    dv=128, dtype="bf16", amp=1.0,
                                                    mask=MASK_CAUSAL_TAIL | MASK_KEY_PADDING,
                                                    len_range=(4096, 8192), layout="bshd"),
}


# Multi-head attention sublayers (projections + attention + output projection)
# of the same three Transformer roles: x, mem ~ N(0, 1); weights ~ N(0, 1/fan_in)
# (unit-variance projections); biases ~ N(0, 0.1^2).
STREAM_X, STREAM_MEM, STREAM_W, STREAM_B = 4, 5, 6, 10  # W: 6..9, b: 10..13 (q, k, v, o)

SUBLAYERS = {
    # Transformer-base encoder self-attention sublayer, key + query padding
    "sublayer_enc_bf16_b256_t64_d512_h8": dict(B=256, T=64, S=64, d_model=512, H=8, H_kv=8,
                                               dk=64, dv=64, mask=MASK_KEY_PADDING |
                                               MASK_QUERY_PADDING, len_range=(8, 64),
                                               cross=False),
    # Transformer-base decoder causal self-attention sublayer
    "sublayer_dec_causal_bf16_b128_t128_d512_h8": dict(B=128, T=128, S=128, d_model=512, H=8,
                                                       H_kv=8, dk=64, dv=64, mask=MASK_CAUSAL,
                                                       len_range=None, cross=False),
    # Transformer-big cross-attention sublayer, source key padding
    "sublayer_cross_bf16_b64_t96_s128_d1024_h16": dict(B=64, T=96, S=128, d_model=1024, H=16,
                                                       H_kv=16, dk=64, dv=64,
                                                       mask=MASK_KEY_PADDING,
                                                       len_range=(16, 128), cross=True),
}


def make_sublayer_inputs(spec: dict, seed: int = 0) -> dict:
    """bf16 bits of x, mem (None for self-attention), W_q, W_k, W_v, W_o, their
    biases, and the key lengths (or None) of a sublayer spec."""
    B, T, S, d = spec["B"], spec["T"], spec["S"], spec["d_model"]
    H, Hkv, dk, dv = spec["H"], spec["H_kv"], spec["dk"], spec["dv"]
    x = tensor(seed, STREAM_X, (B, T, d), "bf16")
    mem = tensor(seed, STREAM_MEM, (B, S, d), "bf16") if spec["cross"] else None
    shapes = [(d, H * dk), (d, Hkv * dk), (d, Hkv * dv), (H * dv, d)]
    w = [tensor(seed, STREAM_W + i, sh, "bf16", amp=float(1.0 / np.sqrt(sh[0])))
         for i, sh in enumerate(shapes)]
    b = [tensor(seed, STREAM_B + i, (sh[1],), "bf16", amp=0.1) for i, sh in enumerate(shapes)]
    lr = spec.get("len_range")
    lens = lengths(seed, B, lr[0], lr[1]) if lr is not None else None
    return dict(x=x, mem=mem, w=w, b=b, lens=lens)


def sublayer_attention_spec(spec: dict) -> dict:
    """The attention step of a sublayer spec, as an attention workload spec."""
    return dict(B=spec["B"], H=spec["H"], Lq=spec["T"], Lk=spec["S"], dk=spec["dk"],
                dv=spec["dv"], dtype="bf16", amp=1.0, mask=spec["mask"],
                len_range=spec.get("len_range"), Hkv=spec["H_kv"], layout="bshd")


def default_scale(dk: int) -> float:
    """1/sqrt(d_k) as the float32 value a caller passes through the C ABI."""
    return float(np.float32(1.0 / np.sqrt(np.float64(dk))))


def make_inputs(spec: dict, seed: int = 0):
    """Q, K, V and key lengths for a workload spec.

    Layout spec["layout"] ("bhsd" [B, heads, L, d], the default, or "bshd"
    [B, L, heads, d]); K and V have spec["Hkv"] heads (default H).
    """
    B, H, Lq, Lk = spec["B"], spec["H"], spec["Lq"], spec["Lk"]
    dk, dv, dt, amp = spec["dk"], spec["dv"], spec["dtype"], spec.get("amp", 1.0)
    Hkv = spec.get("Hkv", H)
    if spec.get("layout", "bhsd") == "bshd":
        qs, ks, vs = (B, Lq, H, dk), (B, Lk, Hkv, dk), (B, Lk, Hkv, dv)
    else:
        qs, ks, vs = (B, H, Lq, dk), (B, Hkv, Lk, dk), (B, Hkv, Lk, dv)
    q = tensor(seed, STREAM_Q, qs, dt, amp)
    k = tensor(seed, STREAM_K, ks, dt, amp)
    v = tensor(seed, STREAM_V, vs, dt, amp)
    lr = spec.get("len_range")
    lens = lengths(seed, B, lr[0], lr[1]) if lr is not None else None
    return q, k, v, lens


# The incoming gradient of the attention output for the backward pass: N(0, 1)
# in the output's layout and dtype (a loss whose gradient is unit-variance noise).
STREAM_DOUT = 14


def make_dout(spec: dict, seed: int = 0) -> np.ndarray:
    """dL/dout for a workload spec: the output's shape and layout, dtype spec["dtype"]."""
    B, H, Lq, dv = spec["B"], spec["H"], spec["Lq"], spec["dv"]
    shape = (B, Lq, H, dv) if spec.get("layout", "bhsd") == "bshd" else (B, H, Lq, dv)
    return tensor(seed, STREAM_DOUT, shape, spec["dtype"])


def as_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of stored values to float64."""
    if dtype == "bf16":
        return bf16_bits_to_f64(x)
    return x.astype(np.float64)
