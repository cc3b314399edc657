"""bench.py's multi-rank bookkeeping on CPU: two gloo ranks (127.0.0.1), each
with its own timing, agree on the max time and the summed launch count, the way
N independent GPU replicas report one whole-job line."""
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


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mx = bench.max_over_ranks(1.5 + rank, world)       # per-rank ms/step
    tot = bench.sum_over_ranks(10.0 * (rank + 1), world)  # per-rank launches
    bench.barrier(world)
    q.put((rank, mx, tot))
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_timing_and_counts():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.5, 2.5]
    assert [r[2] for r in res] == [30.0, 30.0]
