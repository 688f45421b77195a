"""The multi-rank bench path on CPU: two gloo ranks (the GPU job shards decode batches by
rank with no data-path collective; only the timing reduction crosses ranks)."""
import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # each rank times its own replica; the job reports the slowest rank
        ms = [3.0, 5.0][rank]
        m = bench._max_over_ranks(ms, world, torch.device("cpu"))
        rate = bench.whole_job_rate(32 * 10, world, m)
        dist.barrier()
        # the reference arm runs on rank 0 only: other ranks return without work
        if rank == 1:
            class A:
                steps, warmup, gpus = 1, 3, world
            bench.reference_main(A(), rank)
        q.put((rank, m, rate, bench.rank_seed(rank)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_weak_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    for rank, m, rate, seed in out:
        assert m == 5.0                                   # max over ranks
        assert rate == pytest.approx(2 * 320 / 5e-3)      # all ranks' queries / slowest time
    assert out[0][3] != out[1][3]                         # distinct replica inputs per rank


def test_single_rank_passthrough():
    sys.path.insert(0, ROOT)
    import bench
    assert bench._max_over_ranks(4.0, 1, None) == 4.0
    assert bench.whole_job_rate(100, 1, 2.0) == pytest.approx(50_000.0)
