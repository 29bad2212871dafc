"""The multi-rank path of bench.py on CPU (gloo, world size 2): each rank runs
an independent fill, and the whole-job number is every rank's units over the
slowest rank's time. No data-path collective exists; only the timing is reduced."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    ws, r = bench.dist_init("gloo")
    assert (ws, r) == (world, rank)
    bench.barrier()
    # rank 0 processed 1000 units per step in 50 ms, rank 1 the same in 80 ms
    value, ms_per_step, t_max = bench.aggregate_timing(1000, 10, 50.0 if rank == 0 else 80.0)
    out[rank] = (value, ms_per_step, t_max)
    dist.destroy_process_group()


def test_two_rank_timing_reduction_on_gloo():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    for rank in (0, 1):
        value, ms_per_step, t_max = out[rank]
        assert t_max == 80.0
        assert ms_per_step == pytest.approx(8.0)
        assert value == pytest.approx(2 * 1000 * 10 / 0.080)


def test_single_process_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    value, ms, t = bench.aggregate_timing(500, 4, 20.0)
    assert (value, ms, t) == (pytest.approx(100000.0), 5.0, 20.0)
