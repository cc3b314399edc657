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


def test_reference_arm_under_two_ranks():
    """`bench.py --impl reference` launched as two ranks: rank 0 alone runs the
    oracle and prints one JSON line; rank 1 exits 0 without work or output."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2",
                   LOCAL_RANK=str(rank))
        procs.append(subprocess.Popen(
            [sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2",
             "--workload", "tiny-fp32", "--steps", "2", "--warmup", "1", "--oracle-tokens", "16"],
            cwd=root, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=300) for p in procs]
    assert [p.returncode for p in procs] == [0, 0], [o[1][-2000:] for o in outs]
    lines0 = [ln for ln in outs[0][0].splitlines() if ln.startswith("{")]
    assert len(lines0) == 1
    line = json.loads(lines0[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
    assert not [ln for ln in outs[1][0].splitlines() if ln.strip()]
