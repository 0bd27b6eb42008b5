"""The benchmark's N > 1 host logic on CPU with the gloo backend, world size 2: the barrier,
the max-over-ranks timing and the whole-job aggregation of replica throughput."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    r, w, local = bench.dist_setup()
    bench.barrier(w)
    ms = bench.max_over_ranks(1.0 + 2.0 * r, w)  # rank 1 is the slow one
    per_rank_bytes = 1_000_000_000
    value = w * per_rank_bytes / (ms * 1e-3) / 1e9
    q.put((r, w, local, ms, value))
    import torch.distributed as dist

    dist.destroy_process_group()


def test_two_rank_replica_timing():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [x[0] for x in res] == [0, 1] and all(x[1] == 2 for x in res)
    # both ranks see the slowest rank's time; the value counts both replicas' bytes
    assert all(x[3] == 3.0 for x in res)
    assert all(abs(x[4] - 2 * 1.0 / 3e-3) < 1e-9 for x in res)
