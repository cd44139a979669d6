"""The N > 1 bench path's host logic on two gloo ranks (CPU only): timings
are reduced with MAX over ranks and the whole-job rates count every rank's
full workload (weak scaling, independent rows, no data-path collective)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        assert (w, r, local) == (world, rank, rank)
        # each rank reports a different kernel time; the slowest must win
        kernel_ms, region_ms = bench.max_over_ranks([10.0 + rank, 20.0 - rank])
        out[rank] = (kernel_ms, region_ms)
    finally:
        dist.destroy_process_group()


def test_two_rank_max_reduction():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world,
                           start_method="spawn", join=True)
        results = dict(out)
    assert results[0] == results[1] == (11.0, 20.0)


def test_weak_scaling_rates():
    gbs, rows = bench.weak_scaling_rates(world=4, bytes_per_step=8_589_950_976,
                                         rows_per_step=262144, steps=10, slowest_ms=12.9)
    assert gbs == pytest.approx(4 * 8_589_950_976 * 10 / 12.9e-3 / 1e9)
    assert rows == pytest.approx(4 * 262144 * 10 / 12.9e-3)
    g1, _ = bench.weak_scaling_rates(1, 8_589_950_976, 262144, 10, 12.9)
    assert gbs == pytest.approx(4 * g1)
