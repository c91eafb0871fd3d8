"""bench.py's multi-rank arithmetic (one process per GPU, weak scaling): the job
time is the slowest rank's and the value counts every rank's rows.  Run as two
gloo ranks on the CPU."""
import os
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, local = bench.dist_setup()
    ms = [3.0, 5.0][rank]  # rank 1 is the slow one
    t = bench.max_over_ranks(ms, dist, torch.device("cpu"))
    out[rank] = (w, r, local, t, bench.job_rows_per_s(w, 1000, t))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_and_count_all_rows():
    mgr = mp.Manager()
    out = mgr.dict()
    port = 29500 + os.getpid() % 1000
    mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
    assert out[0][:3] == (2, 0, 0) and out[1][:3] == (2, 1, 1)
    for r in (0, 1):
        assert out[r][3] == 5.0
        assert out[r][4] == pytest.approx(2 * 1000 / 0.005)


def test_single_rank_without_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.0, None, None) == 4.0
    assert bench.job_rows_per_s(1, 262144, 4.0) == pytest.approx(262144 / 0.004)
