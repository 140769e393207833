"""The multi-rank bench logic on CPU with two gloo ranks: each rank gets its
own batch (weak scaling), the step time is the slowest rank's, and the job
throughput counts every rank's bytes."""
import os

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from paged_kv_cache_220_gb300 import synth, workload


def _rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = workload.rank_workload(synth.tiny(), rank, world)
        seeds = [None] * world
        dist.all_gather_object(seeds, w.seed)
        ms = workload.max_over_ranks(10.0 + rank * 5.0, dist)
        dist.barrier()
        q.put((rank, seeds, ms, workload.job_throughput(10 ** 9, world, ms)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29517
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    out.sort()
    (_, seeds0, ms0, v0), (_, seeds1, ms1, v1) = out
    assert seeds0 == seeds1 and seeds0[0] != seeds0[1]        # distinct batches
    assert ms0 == ms1 == 15.0                                  # the slowest rank
    assert abs(v0 - 2 * 1e9 / 0.015 / 1e9) < 1e-9              # both ranks' bytes


def test_single_rank_is_identity():
    w = synth.tiny()
    assert workload.rank_workload(w, 0, 1) is w
    assert workload.max_over_ranks(3.5) == 3.5
