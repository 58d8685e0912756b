"""bench.py's replica aggregation across ranks, on CPU with gloo (world size 2):
each timed region is the max over ranks and the bytes are summed."""
import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    cpu = torch.device("cpu")
    t = bench.reduce_max(10.0 + rank * 5.0, cpu)
    b = bench.reduce_sum(1000.0 * (rank + 1), cpu)
    # per-region times: the max over ranks of each region, then the median
    regions = bench.reduce_max_list([1.0 + rank, 5.0 - rank, 3.0], cpu)
    bench.barrier()
    q.put((rank, t, b, tuple(regions)))
    dist.destroy_process_group()


def test_max_time_and_summed_bytes_over_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 15.0, 3000.0, (2.0, 5.0, 3.0)), (1, 15.0, 3000.0, (2.0, 5.0, 3.0))]


def test_single_process_is_identity():
    import bench
    assert bench.reduce_max(3.5, torch.device("cpu")) == 3.5
    assert bench.reduce_sum(7.0, torch.device("cpu")) == 7.0
    assert bench.reduce_max_list([1.0, 2.0], torch.device("cpu")) == [1.0, 2.0]
