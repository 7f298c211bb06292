"""The N > 1 path of bench.py runs independent replicas (batch-1 drafting does
not shard without tensor parallelism): a barrier around the timed region, the
slowest rank's time, and a whole-job value of N cycles per step.  Checked with
two gloo ranks on the CPU (no GPU, no data-path collective)."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    local_ms = 1.0 + 0.5 * rank          # rank 1 is the slow one
    slow = bench.max_over_ranks(local_ms, world)
    bench.barrier(world)
    out[rank] = (slow, bench.replica_value(slow, world))
    # the reference arm runs on rank 0 only; other ranks return without work
    if rank != 0:
        assert bench.run_reference(None, rank, world) is None
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world, port = 2, _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1] == (1.5, pytest.approx(2 * 1e3 / 1.5))


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.replica_value(2.0, 1) == 500.0
