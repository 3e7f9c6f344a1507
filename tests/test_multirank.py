"""Multi-rank logic of bench.py on CPU (gloo, world_size 2): the slowest
rank's time decides, and the whole-job value counts every rank's work.  The
(batch, head) pairs are independent, so ranks exchange nothing but timings."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import gen
        w, r, lr = bench.dist_env()
        mine = 0.010 + 0.005 * rank  # rank 1 is slower
        slowest = bench.max_over_ranks(mine, w)
        spec = gen.WORKLOADS["dec_causal_bf16_b128_h8_l128_d64"]
        nbytes, flops = bench.algorithmic(spec, None)
        value = bench.weak_scaling_value(spec, nbytes, flops, slowest, w)
        bench.barrier(w)
        q.put((r, w, lr, slowest, value, nbytes))
    finally:
        dist.destroy_process_group()


def test_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for r, (rank, world, local, slowest, value, nbytes) in enumerate(res):
        assert (rank, world, local) == (r, 2, r)
        assert slowest == pytest.approx(0.015)
        assert value == pytest.approx(2 * nbytes / 0.015 / 1e9)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(0.25, 1) == 0.25
