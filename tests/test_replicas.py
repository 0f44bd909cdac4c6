"""The multi-GPU path is replicas only (each rank runs its own copy of the workload,
weak scaling): the one cross-rank step is the timing aggregate, the slowest rank's time
and the sum of every rank's units.  Checked with world-size-2 gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import sys
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms, units = bench.replica_aggregate(10.0 + 5.0 * rank, 1000.0 * (rank + 1), dist, "cpu")
    q.put((rank, ms, units))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_replica_aggregate_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, units in got:
        assert ms == 15.0                        # the slowest rank's time, on every rank
        assert units == 3000.0                   # every rank's units
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.replica_aggregate(7.5, 42.0) == (7.5, 42.0)      # one process: no collective
