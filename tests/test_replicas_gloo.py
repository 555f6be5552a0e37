"""bench.py's multi-rank host logic on CPU: two gloo ranks, the barrier and the
max-over-ranks timing that turns per-rank replica times into one job time."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    r, w, _ = bench.dist_setup(world)
    bench.barrier(w)
    t_rank = 1.0 + 0.5 * r                   # a per-rank replica time
    t_job = bench.reduce_max(t_rank, w)
    tokens = 7 * 3 * w                       # T * K per rank, all ranks
    q.put((r, w, t_job, tokens / t_job))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[0] for r in res] == [0, 1]
    for _, w, t_job, value in res:
        assert w == 2
        assert t_job == pytest.approx(1.5)
        assert value == pytest.approx(42 / 1.5)
