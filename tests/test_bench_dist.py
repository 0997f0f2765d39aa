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


def test_algorithmic_work_of_the_bf16_and_fp8_layers():
    """The per-launch work bench.py divides by its timings: the flops of the formulas and
    the least bytes each stage moves, in bf16 and with e4m3 rows, W13, h and W2."""
    import bench
    from routing_dispatch_combine_moe_b300 import workloads as wl
    W = wl.WORKLOADS
    T, d, E, k, F = 2048, 4096, 8, 2, 14336
    rows = T * k
    bf = bench.algorithmic(W["mixtral_bf16"], rows, out_bytes=4, h_cols=F)
    assert bf["up_flops"] == 2 * rows * d * 2 * F and bf["down_flops"] == 2 * rows * F * d
    assert bf["up_bytes"] == E * 2 * F * d * 2 + rows * d * 2 + rows * F * 2
    assert bf["down_bytes"] == E * d * F * 2 + rows * F * 2 + rows * d * 4
    # the combine's algorithmic bytes take the activation dtype; the fp32 expert rows it
    # actually reads are counted apart
    assert bf["combine_bytes"] == rows * d * 2 + T * d * 2
    assert bf["combine_bytes_moved"] == rows * d * 4 + T * d * 2
    # experts without rows are skipped: only the active experts' weights count
    six = bench.algorithmic(W["mixtral_bf16"], rows, out_bytes=4, h_cols=F, active_experts=6)
    assert bf["up_bytes"] - six["up_bytes"] == 2 * 2 * F * d * 2 and bf["down_bytes"] - six["down_bytes"] == 2 * d * F * 2
    assert six["up_flops"] == bf["up_flops"]
    # the DeepSeek-V3-shaped layer: x read, rows written, rows read, y written = 1057 MB
    ds = bench.algorithmic(W["dsv3_full"], 4096 * 8, out_bytes=4, h_cols=2048)
    assert ds["dispatch_bytes"] + ds["combine_bytes"] == 2 * (4096 + 32768) * 7168 * 2 == 1_056_964_608
    f8 = bench.algorithmic(W["mixtral_fp8_gemm"], rows, out_bytes=4, h_cols=F)
    assert f8["up_flops"] == bf["up_flops"] and f8["down_bytes"] == bf["down_bytes"]
    # e4m3 W13 with one scale per row, rows as d codes + one scale, h still bf16
    assert f8["up_bytes"] == E * 2 * F * (d + 4) + rows * (d + 4) + rows * F * 2
    # the dispatch writes codes + a scale per row instead of bf16 rows
    assert f8["dispatch_bytes"] - bf["dispatch_bytes"] == rows * (d + 4) - rows * d * 2
    both = bench.algorithmic(W["mixtral_fp8_experts"], rows, out_bytes=4, h_cols=F)
    # the down stage reads bf16 h, writes and reads its codes + scales, reads e4m3 W2
    assert both["down_bytes"] == E * d * (F + 4) + rows * F * 2 + 2 * rows * (F + 4) + rows * d * 4
    assert bench.fp8_row_bytes(4096) == 4096 + 4 * 32 and bench.fp8_row_bytes(4096, per_row=True) == 4100
    # deduplicated FP8 send rows: x read once, each send row written and read as codes +
    # block scales, each expert row written in bf16
    T2, d2, rows2, sent = 4096, 7168, 32768, 16000
    ddf = bench.algorithmic(W["dsv3_grouped_dedup_fp8"], rows2, out_bytes=2, h_cols=0, rows_sent=sent)
    assert ddf["dispatch_bytes"] == T2 * d2 * 2 + rows2 * d2 * 2 + 2 * sent * (d2 + 4 * 56)
    # deduplicated send rows in the FP8 GEMM's format: codes + one scale, and so the expert rows
    ddg = bench.algorithmic(W["dsv3_full_fp8_gemm_dedup"], rows2, out_bytes=4, h_cols=2048, rows_sent=sent)
    assert ddg["dispatch_bytes"] == T2 * d2 * 2 + rows2 * (d2 + 4) + 2 * sent * (d2 + 4)
