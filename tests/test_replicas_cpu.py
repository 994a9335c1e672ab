"""The multi-GPU path of the benchmark on CPU: two gloo ranks in spawned
processes.

The layer does not shard (one GPU's experts, no exchange step), so `bench.py
--gpus N` runs N independent replicas: rank 0 builds the shared in-tree library
while the others wait at a barrier, every rank times its own replica, and the
job's time is the slowest rank's.  The reference arm runs on rank 0 only; the
other ranks leave without work or output.  No GPU is touched."""
import contextlib
import io
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


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from dropless_mixture_experts_top_gb300 import _build
    built = []
    _build.build = lambda *a, **k: built.append(rank)  # record who builds; build nothing
    bench.ensure_built(rank, dist)
    slowest = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")
    out = io.StringIO()
    rc = None
    if rank != 0:  # the reference arm: only rank 0 runs the oracle and prints
        class Args:
            steps, warmup, workload, tokens, gpus = 1, 3, bench.DEFAULT_WORKLOAD, 0, world
        with contextlib.redirect_stdout(out):
            rc = bench.run_reference(Args())
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, built, slowest, rc, out.getvalue()))


def test_two_gloo_replicas():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in procs:
        rank, built, slowest, rc, out = q.get(timeout=120)
        res[rank] = (built, slowest, rc, out)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][0] == [0] and res[1][0] == []   # rank 0 alone builds
    assert res[0][1] == res[1][1] == 15.0         # both see the slowest rank's time
    assert res[1][2] == 0 and res[1][3] == ""     # the reference arm leaves rank 1 without work
