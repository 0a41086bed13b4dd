"""The N > 1 path of bench.py on CPU: two gloo ranks (world_size 2, 127.0.0.1).

Each rank runs its own batch (weak scaling); the only collective is the max
over ranks of the timing, and the reported value is the units all ranks
processed divided by that time.  No GPU and no data-path collective is involved.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    ms = [3.0, 5.0][rank]                       # rank 1 is the slower one
    out[rank] = bench.max_over_ranks(ms, w)
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == 5.0
    # whole-job value: units of both ranks over the slowest rank's time
    import bench
    steps, units = 10, 16384
    assert 2 * steps * units / (out[0] * 1e-3) == pytest.approx(2 * 10 * 16384 / 0.005)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5, 1) == 7.5
    bench.barrier(1)
