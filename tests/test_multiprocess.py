"""N > 1 host logic on CPU: world_size-2 gloo process groups.

Each rank of bench.py runs an independent replica of the workload (the path
has no exchange step); the only cross-rank steps are the barrier and the
max-over-ranks of the timed region, checked here, and the reference arm's
rule that ranks other than 0 do no work."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mx = bench.reduce_max(10.0 + 5 * rank, "cpu", world)
    dist.barrier()

    class A:
        workload = "tiny"
        steps = 1
        warmup = 3
    ref = bench.run_reference(A()) if rank != 0 else "skipped"
    q.put((rank, mx, ref))
    dist.destroy_process_group()


def test_reduce_max_and_reference_rank_rule_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    assert out[0][1] == out[1][1] == 15.0
    assert out[1][2] is None          # rank 1 of the reference arm does no work
