"""The allocation-free sublayer entry point (mha_sublayer_fwd_static) against
the workspace entry point (mha_sublayer_fwd), on the GPU.

This file is collected last so that it also runs after every other GPU test;
it must pass alone as well.  Two calls in a row through each entry point give
the same bits, whatever the static scratch held before.
"""
import gc
import math

import numpy as np
import pytest

import gen
from helpers import from_device, to_device

pytestmark = pytest.mark.gpu


def _inputs(B, T, S, d, H, H_kv, mask, cross, seed):
    rng = np.random.default_rng(seed)
    dk = d // H
    bf = gen.f64_to_bf16_bits
    x = bf(rng.normal(size=(B, T, d)))
    mem = bf(rng.normal(size=(B, S, d))) if cross else None
    w = [bf(rng.normal(size=(d, n)) / math.sqrt(d)) for n in (H * dk, H_kv * dk, H_kv * dk)]
    w.append(bf(rng.normal(size=(H * dk, d)) / math.sqrt(H * dk)))
    b = [bf(rng.normal(size=n) * 0.1) for n in (H * dk, H_kv * dk, H_kv * dk, d)]
    lens = rng.integers(1, S + 1, size=B).astype(np.int32) if mask & 6 else None
    return x, mem, w, b, lens


@pytest.mark.parametrize("B,T,S,d,H,H_kv,mask,cross", [
    (8, 64, 64, 512, 8, 8, gen.MASK_KEY_PADDING | gen.MASK_QUERY_PADDING, False),
    (4, 96, 128, 1024, 16, 4, gen.MASK_KEY_PADDING, True),
    (2, 200, 200, 512, 8, 8, gen.MASK_CAUSAL, False),
])
def test_static_scratch_matches_workspace_entry_point(B, T, S, d, H, H_kv, mask, cross):
    import torch
    import transformer_head_scaled_mha_gb300 as mha
    x, mem, w, b, lens = _inputs(B, T, S, d, H, H_kv, mask, cross, seed=B + T + d)
    dev = lambda a: to_device(a, "bf16") if a is not None else None
    kl = torch.from_numpy(lens).cuda() if lens is not None else None
    args = (dev(x), *[dev(t) for t in w], *[dev(t) for t in b])
    kw = dict(mem=dev(mem), H=H, H_kv=H_kv, mask_kind=mask, key_lengths=kl)
    ref = [from_device(mha.mha_sublayer_fwd(*args, **kw)) for _ in range(2)]
    got = [from_device(mha.mha_sublayer_fwd_static(*args, **kw)) for _ in range(2)]
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ref[0], ref[1])
    np.testing.assert_array_equal(got[0], ref[0])
    np.testing.assert_array_equal(got[1], ref[0])
    assert mha.mha_debug_status() == mha.MHA_OK


def test_static_scratch_refuses_shapes_beyond_it():
    import torch
    import transformer_head_scaled_mha_gb300 as mha
    x = torch.zeros(257, 64, 512, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(512, 512, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mha.MhaError) as e:
        mha.mha_sublayer_fwd_static(x, w, w, w, w, H=8)
    assert e.value.status == mha.MHA_ERR_UNSUPPORTED


def test_static_entry_point_allocates_no_device_memory():
    """After a first call (which loads the kernels' code and looks the scratch
    up), further calls through the C entry point leave the device's free
    memory, and everything the caching allocator holds, exactly as they were."""
    import ctypes

    import torch
    import transformer_head_scaled_mha_gb300 as mha
    B, T, d, H = 8, 64, 512, 8
    x, _, w, b, lens = _inputs(B, T, T, d, H, H, gen.MASK_KEY_PADDING | gen.MASK_QUERY_PADDING,
                               False, seed=7)
    dev = lambda a: to_device(a, "bf16")
    xd, wd, bd = dev(x), [dev(t) for t in w], [dev(t) for t in b]
    kl = torch.from_numpy(lens).cuda()
    out = torch.empty((B, T, d), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    p = lambda t: ctypes.c_void_p(t.data_ptr())

    def call():
        return mha.lib.mha_sublayer_fwd_static(
            p(xd), None, p(out), *[p(t) for t in wd], *[p(t) for t in bd], B, T, T, d, H, H,
            d // H, d // H, gen.MASK_KEY_PADDING | gen.MASK_QUERY_PADDING, p(kl),
            ctypes.c_float((d // H) ** -0.5), mha.MHA_DTYPE_BF16,
            ctypes.c_void_p(stream.cuda_stream))

    assert call() == mha.MHA_OK
    torch.cuda.synchronize()
    first = from_device(out)
    # tensors left by earlier tests must not be freed in between (that would
    # move the caching allocator's counters without any call of ours)
    gc.collect()
    gc.disable()
    try:
        before = (torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated(),
                  torch.cuda.memory_reserved())
        for _ in range(2):
            assert call() == mha.MHA_OK
        torch.cuda.synchronize()
        after = (torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated(),
                 torch.cuda.memory_reserved())
    finally:
        gc.enable()
    assert after == before
    np.testing.assert_array_equal(from_device(out), first)
    assert mha.mha_debug_status() == mha.MHA_OK
