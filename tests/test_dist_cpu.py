"""The multi-rank path of bench.py on CPU: two gloo ranks (replicas only).

The decode path has no exchange step, so N GPUs run N independent batches; the
host logic that remains -- rendezvous on 127.0.0.1, a barrier, the max of the
ranks' times and the sum of their bytes (weak scaling) -- runs here with the gloo
backend, world size 2."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench
    w, r, lr = bench.dist_env()
    dist = bench.dist_init(w, "gloo")
    bench.barrier(dist)
    ms = bench.max_over_ranks(dist, 10.0 + rank)           # slowest rank's time
    total = bench.sum_over_ranks(dist, 1000.0 * (rank + 1))  # bytes of all ranks
    # the reference arm runs on rank 0 only; other ranks return without work
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "1"])
    ref = bench.run_reference(args) if rank != 0 else "skipped"
    dist.destroy_process_group()
    q.put((rank, w, r, ms, total, ref))


def test_two_gloo_ranks_weak_scaling_host_logic():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, w, r, ms, total, ref in res:
        assert w == 2 and r == rank
        assert ms == 11.0            # max over ranks
        assert total == 3000.0       # sum over ranks
    assert res[1][5] is None         # rank 1 of the reference arm does no work


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.dist_init(1, "gloo") is None
    assert bench.max_over_ranks(None, 3.5) == 3.5
    assert bench.sum_over_ranks(None, 2.0) == 2.0
