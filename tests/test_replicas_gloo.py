"""The N > 1 path of bench.py on CPU: world_size 2 over gloo (127.0.0.1).

The scan does not shard: N GPUs run N independent replicas, and the only cross-rank steps are
the barrier around the timed region and the maximum of the ranks' times. These tests run those
helpers in two real processes with different local times and check that both ranks see the
slowest one, and that the whole-job throughput counts every replica's units.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    ws, r, _ = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=ws)
    dist.barrier()
    m = bench.max_over_ranks(dist, times[r], "cpu")
    out[r] = (m, bench.job_throughput(1000.0, ws, m))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_both_replicas():
    world, port = 2, _free_port()
    times = [0.25, 0.40]
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        m, thr = res[r]
        assert m == max(times)
        assert thr == pytest.approx(2 * 1000.0 / max(times))


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, 1.5, "cpu") == 1.5
    assert bench.job_throughput(10.0, 1, 2.0) == 5.0
