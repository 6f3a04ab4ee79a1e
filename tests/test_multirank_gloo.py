"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

Each rank is an independent replica (no collective on the data path); the
only cross-rank operations are the barrier and the max-over-ranks of the
timed region, which these tests exercise without a GPU.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, times, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_env()
    bench.barrier(w)
    m = bench.max_over_ranks(times[r], w, device="cpu")
    v = bench.job_throughput(65536, 10, w, m)
    q.put((r, lr, m, v))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("times", [(100.0, 250.0), (300.0, 120.0)])
def test_max_over_ranks_and_job_throughput(times):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    mx = max(times)
    for r, lr, m, v in res:
        assert r == lr and m == mx
        assert abs(v - 65536 * 2 * 10 / (mx / 1e3)) < 1e-6 * v


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(100, 2, 1, 1000.0) == 200.0
