"""The N > 1 launch path of bench.py, exercised with two gloo ranks on the CPU.

The GMA forward shards by independent (batch, head) units, so several GPUs run independent
replicas with no collective on the data path; the only cross-rank steps are the barrier around the
timed region and the maximum of the per-rank step times.  Those run here over gloo.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_setup() == (world, rank, rank)
    dist.barrier()
    ms = [3.0, 5.0][rank]  # the slower rank sets the job's step time
    m = bench.max_over_ranks(ms, world)
    out[rank] = (m, bench.whole_job_rate(1000, m, world))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step_time():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    m, rate = res[0]
    assert m == 5.0
    assert rate == pytest.approx(2 * 1000 / 5e-3)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.whole_job_rate(10, 2.0, 1) == pytest.approx(5000.0)
