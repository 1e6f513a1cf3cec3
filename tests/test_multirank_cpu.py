"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

Each rank runs its own replica of the workload (weak scaling, no collective
on the data path); the job's throughput is all ranks' units divided by the
slowest rank's time.  Two gloo ranks with different timings check that
every rank sees the same maximum and the same whole-job value.
"""
import os
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    secs = [0.25, 0.40][rank]
    mx = bench.max_over_ranks(secs, world, "cpu")
    val = bench.whole_job_value(1000.0, world, mx)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, mx, val))


def test_two_gloo_ranks_agree_on_max_time_and_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for _, mx, val in res:
        assert mx == pytest.approx(0.40)
        assert val == pytest.approx(2 * 1000.0 / 0.40)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.3, 1, "cpu") == 0.3
    assert bench.whole_job_value(10.0, 1, 0.5) == 20.0
