"""The give-up path of the kernels' bounded waits, on the GPU, without any
fault: a test hook makes the MMA issuer wait on a barrier that nothing
signals, with a wait limit of 2 ms.  The kernel must then let its copies and
products in flight finish, free its tensor memory, report MHA_ERR_TIMEOUT
through the status word (cleared by the read), and leave the context usable:
the next normal call matches the oracle.

Packed short-sequence kernel: the stall comes before the first product, with
every CTA's first copies in flight.  Long-sequence kernel: before the third
key tile, with products and copies of the first two in flight.
"""
import numpy as np
import pytest

import gen
from helpers import check_case, run_gpu, spec

pytestmark = pytest.mark.gpu

STALL_SHORT, STALL_LONG = 1, 2


@pytest.mark.parametrize("stall,case,path", [
    (STALL_SHORT, spec(4, 2, 64, 64, 64, mask=gen.MASK_KEY_PADDING | gen.MASK_QUERY_PADDING,
                       len_range=(8, 64)), 2),
    (STALL_SHORT, spec(3, 4, 128, 128, 64, mask=gen.MASK_CAUSAL), 2),
    (STALL_LONG, spec(1, 2, 512, 512, 128, mask=gen.MASK_CAUSAL, amp=0.5), 3),
    (STALL_LONG, spec(2, 2, 600, 600, 64), 3),
])
def test_a_wait_that_runs_out_reports_timeout_and_recovers(stall, case, path):
    import torch
    import transformer_head_scaled_mha_gb300 as mha
    assert mha.mha_fwd_path_ex(case["B"], case["H"], case["Hkv"], case["Lq"], case["Lk"],
                               case["dk"], case["dv"], case["mask"], 1) == path
    q, k, v, lens = gen.make_inputs(case, seed=3)
    assert mha.mha_debug_status() == mha.MHA_OK
    assert mha.mha_debug_set_wait(2_000_000, stall) == mha.MHA_OK
    try:
        run_gpu(q, k, v, lens, case)  # output undefined: the kernel gave up
        torch.cuda.synchronize()
    finally:
        assert mha.mha_debug_set_wait(0, 0) == mha.MHA_OK
    assert mha.mha_debug_status() == mha.MHA_ERR_TIMEOUT
    assert mha.mha_debug_status() == mha.MHA_OK  # the read cleared it
    # the same call with the default limit and no stall: correct, status clean
    check_case(case, seed=3, label="after a give-up")
    assert mha.mha_debug_status() == mha.MHA_OK
