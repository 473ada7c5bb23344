"""Several GPUs run independent replicas of the pass (the path has no exchange
step): the job's time is the slowest rank's and its work the sum over ranks.
Checked with two gloo ranks on the CPU."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    times = [10.0 + rank, 20.0 - rank]
    counts = [100 * (rank + 1), 7]
    t, c = bench.over_ranks(times, counts, world)
    out[rank] = (t, c)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_max_time_and_sum_work():
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        t, c = res[rank]
        assert t == [11.0, 20.0]
        assert c == [300.0, 14.0]


def test_single_rank_is_unchanged():
    import bench
    assert bench.over_ranks([3.0], [5], 1) == ([3.0], [5.0])
