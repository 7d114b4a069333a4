"""Host logic of the multi-GPU benchmark on CPU (gloo, world size 2).

The attention path has no exchange step, so N GPUs run N independent
replicas; the only collective is the max of the timed region over ranks,
and the whole-job number is N x bytes per step x steps / that max."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, l = bench.dist_setup()
    ms = 10.0 + 5.0 * rank                      # rank 1 is the slow replica
    m = bench.max_over_ranks(ms, "cpu")
    out[rank] = (w, r, l, m, bench.replica_throughput(4e9, 100, m, w))
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank():
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    for rank in range(2):
        w, r, l, m, gbs = out[rank]
        assert (w, r, l) == (2, rank, rank)
        assert m == 15.0
        assert gbs == pytest.approx(2 * 4e9 * 100 / 0.015 / 1e9)


def test_single_process_needs_no_collective():
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.replica_throughput(1e9, 10, 1000.0, 1) == pytest.approx(10.0)
