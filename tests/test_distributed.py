"""The multi-rank bench logic on CPU: two gloo ranks, each with its own
replica of the workload (different seeds, no data-path collective), and the
timing aggregation (max of times, sum of bytes) over ranks."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    import pkv_workloads as wl

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank owns a different replica of the batch
        b = wl.decode_batch(wl.LONG_GQA_8K, seed=rank, batch=2, ctx_override=[40 + rank, 17])
        lens = b.context_lens.tolist()
        t = bench.reduce_max(float(rank + 1) * 1.5, world, torch.device("cpu"))
        s = bench.reduce_sum(float(sum(lens)), world, torch.device("cpu"))
        bench.barrier(world)
        q.put((rank, lens, float(b.q.float().sum()), t, s))
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_and_timing_reduction():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, lens0, qs0, t0, s0), (r1, lens1, qs1, t1, s1) = res
    assert lens0 == [40, 17] and lens1 == [41, 17]
    assert qs0 != qs1                         # independent replicas
    assert t0 == t1 == 3.0                    # max over ranks
    assert s0 == s1 == float(sum(lens0) + sum(lens1))
