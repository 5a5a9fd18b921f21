"""The multi-GPU path of bench.py is replicas only: each rank runs its own
block forward and the job reports the units of all ranks over the slowest
rank's time.  This checks that aggregation with two gloo ranks on the CPU
(no GPU, no collective on the data path)."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [120.0, 150.0][rank]          # the slower rank decides
    ms = bench.max_over_ranks(local_ms, world)
    value = bench.replica_throughput(32768 * 4 * 10, world, ms)
    out[rank] = (ms, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_as_replicas():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 150.0
    expect = 32768 * 4 * 10 * 2 / 0.150
    assert res[0][1] == pytest.approx(expect)
    assert res[1][1] == pytest.approx(expect)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(42.0, 1) == 42.0
    assert bench.replica_throughput(1000, 1, 500.0) == pytest.approx(2000.0)
