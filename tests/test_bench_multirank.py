"""The benchmark's multi-rank aggregation on CPU: two gloo ranks, the timed
interval is the maximum over ranks and the job value counts every rank's
work (replicas only, no data-path collective)."""
import os

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms = [3.0, 5.0][rank]
    total = bench.max_over_ranks(ms, dist, "cpu")
    q.put((rank, total, bench.whole_job_tflops(1e12, world, total)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, total, value in res:
        assert total == 5.0
        assert value == pytest.approx(2 * 1e12 / 5e-3 / 1e12)
