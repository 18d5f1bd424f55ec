"""The bench's N>1 path on CPU: two gloo ranks run the same setup, barrier
and max-over-ranks timing reduction that torchrun ranks run on GPUs (each
rank is an independent replica; no data moves between ranks)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    w, r, local = bench.dist_setup("gloo")
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    t = bench.max_over_ranks(10.0 + 5.0 * rank, w, "cpu")
    out[rank] = t
    dist.destroy_process_group()


def test_two_rank_timing_reduction():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True,
                       start_method="spawn")
    assert out[0] == out[1] == 15.0  # every rank sees the slowest rank's time


def test_aggregate_is_whole_job():
    # 2 ranks x 10 steps x 1e9 bytes in 5 ms (slowest rank) = 4000 GB/s
    assert bench.aggregate_throughput(1e9, 10, 5.0, 2) == pytest.approx(4000.0)
    assert bench.aggregate_throughput(1e9, 10, 5.0, 1) == pytest.approx(2000.0)
