"""Host-side logic of the multi-rank bench path, run as two gloo ranks on the
CPU (one process per GPU on a GPU node; here no GPU is needed): the
rendezvous, the barrier, the max-over-ranks time and the whole-job rate of a
weak-scaling run (every rank processes its own batch, no data collective)."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    w, r, _ = bench.dist_setup(world)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    ms = bench.max_over_ranks(w, 1.0 + 0.5 * r)  # rank 1 is the slow one
    q.put((r, w, ms, bench.job_rate(w, 100.0, ms)))
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    import torch
    import torch.multiprocessing as mp
    if torch.cuda.is_available():
        pytest.skip("exercises the CPU (gloo) path")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    assert [r[0] for r in res] == [0, 1]
    for _, world, ms, rate in res:
        assert world == 2
        assert ms == 1.5  # the max over ranks
        assert rate == pytest.approx(2 * 100.0 / 1.5e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1, 0.25) == 0.25
    assert bench.job_rate(1, 10.0, 2.0) == pytest.approx(5000.0)
