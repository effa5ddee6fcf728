"""The multi-GPU path is replicas: one process per GPU, no collective on the
data path, the job timed by its slowest rank and credited with every rank's
bytes.  Checked here with two gloo ranks on CPU."""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r ran 1 + r seconds and moved 100 (r + 1) bytes
        q.put((rank, *bench.aggregate_replicas(1.0 + rank, 100 * (rank + 1), world)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_replica_aggregation_takes_slowest_rank_and_all_bytes(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for _, secs, nbytes in results:
        assert secs == float(world)                       # max over ranks
        assert nbytes == sum(100 * (r + 1) for r in range(world))


def test_single_rank_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate_replicas(1.5, 42, 1) == (1.5, 42)
