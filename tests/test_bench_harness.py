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


def test_repeats_fill_the_sampled_time():
    sys.path.insert(0, ROOT)
    import bench

    # at least the minimum count; more when regions are short
    assert bench.repeat_count(0.5, 21, 1.5) == 21
    assert bench.repeat_count(0.003, 21, 1.5) == 500
    assert bench.repeat_count(1e-6, 21, 1.5, cap=5000) == 5000
    assert bench.repeat_count(0.0, 21, 1.5) == 21
    s = bench.summarize_regions([3.0, 1.0, 2.0, 10.0, 4.0], 10)
    assert s["repeats"] == 5 and s["median_ms"] == 3.0 and s["min_ms"] == 1.0 and s["max_ms"] == 10.0
    assert s["ms_per_step"] == 0.3
