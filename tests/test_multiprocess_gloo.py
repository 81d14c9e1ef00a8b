"""World-size-2 checks of the bench's multi-rank logic on CPU (gloo): each rank draws its own
batch, the slowest rank's time is what every rank sees, and the whole-job rate aggregates all
ranks' work over that time.  The attention path itself needs no exchange between ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_env()
        my_time = 1.0 + rank  # rank 1 is slower
        t = bench.reduce_max(my_time)
        rate = bench.aggregate_rate(100.0, w, t)
        seed = bench.rank_seed(r)
        from attention_attn_prefill_02_gb300 import synthetic
        x = synthetic.normal((4, 8), seed)
        gathered = [torch.zeros(4, 8) for _ in range(w)]
        dist.all_gather(gathered, x.float())
        q.put((r, w, t, rate, [g.sum().item() for g in gathered]))
    finally:
        dist.destroy_process_group()


def test_two_rank_reduction_and_independent_batches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    for r, w, t, rate, sums in res:
        assert w == 2
        assert t == 2.0                    # the slowest rank's time, seen by every rank
        assert rate == pytest.approx(100.0 * 2 / 2.0)
        assert sums[0] != sums[1]          # the ranks drew different batches
