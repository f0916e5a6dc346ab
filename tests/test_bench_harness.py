"""The multi-rank side of bench.py on CPU (gloo, 2 ranks): each rank times its
own batch of frames (no collective on the data path); the job's time is the
slowest rank's, and the throughput counts every rank's frames."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    r, w, local = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    slowest = bench.reduce_max(10.0 + 5.0 * rank, dist)
    out[rank] = (r, w, local, slowest, bench.job_throughput(w, 32, 100, slowest))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert sorted(res) == [0, 1]
    for rank, (r, w, local, slowest, thr) in res.items():
        assert (r, w, local) == (rank, 2, rank)
        assert slowest == 15.0
        assert thr == 2 * 32 * 100 / 15.0


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.reduce_max(3.5) == 3.5
    assert bench.job_throughput(1, 32, 10, 2.0) == 160.0
