"""bench.py's multi-GPU mode runs independent replicas (slots never interact, so there
is no data-path collective); the host side only meets at barriers and takes the
slowest rank's time.  That host logic runs here as two gloo ranks on the CPU."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    r, w = bench.dist_setup(world)
    assert (r, w) == (rank, world)
    bench.barrier(w)
    slowest = bench.max_over_ranks(10.0 + rank, w)   # rank 1 is the slow one
    bench.barrier(w)
    out.put((rank, slowest))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_replicas_agree_on_the_slowest_time():
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
    assert got == [(0, 11.0), (1, 11.0)]
