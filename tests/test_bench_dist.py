"""The multi-rank path of bench.py on CPU: two gloo ranks, each reporting its
own time and bytes; every rank must get the max of the times and the sum of
the bytes (weak scaling: value = all ranks' bytes / slowest rank's time)."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    assert bench.dist_env() == (world, rank, rank)
    ms, nbytes = bench.aggregate(10.0 + 5 * rank, 1000.0 * (rank + 1))
    bench.barrier()
    q.put((rank, ms, nbytes))
    dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 15.0, 3000.0), (1, 15.0, 3000.0)]


def test_aggregate_single_process_is_identity():
    import bench
    assert bench.aggregate(3.5, 7.0) == (3.5, 7.0)
