"""The benchmark's multi-rank logic on CPU: two gloo ranks, barrier, max over ranks,
whole-job throughput. (On GPUs each rank runs an independent replica of the layer.)"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch
    import bench
    w, r, l = bench.dist_env()
    bench.init_dist(w, l, backend="gloo")
    bench.barrier(w)
    slowest = bench.reduce_max(1.0 + rank, w, torch.device("cpu"))
    value = bench.job_throughput(2048, 10, w, slowest)
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((rank, w, slowest, value))


def test_two_gloo_ranks_take_the_slowest_rank_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, world, slowest, value in res:
        assert world == 2
        assert slowest == pytest.approx(2.0)
        assert value == pytest.approx(2048 * 10 * 2 / 2.0)
