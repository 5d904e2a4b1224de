"""The multi-replica path of bench.py on CPU.  The decode step does not shard:
`--gpus N` runs N independent replicas, and the ranks only agree on the
timing.  Two gloo ranks run the same aggregation as the GPU ranks: the
timed region is the slowest rank's (all_reduce MAX), the value all ranks'
frames over it."""
import os
import socket

import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms, value = bench.replica_timing([100.0, 250.0][rank], 64, dist, "cpu")
    dist.barrier()
    q.put((rank, ms, value))
    dist.destroy_process_group()


def test_replica_timing_two_ranks():
    import torch.multiprocessing as mp
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(60)
    assert [p.exitcode for p in procs] == [0, 0]
    for rank, ms, value in res:
        assert ms == 250.0  # the slowest rank's time, seen by both
        assert value == pytest.approx(world * 64 / 0.25)


def test_replica_timing_single_rank():
    import bench
    ms, value = bench.replica_timing(50.0, 10)
    assert ms == 50.0 and value == pytest.approx(200.0)
