"""The multi-process path of bench.py on CPU (gloo, world size 2): process-group
set-up from the torchrun environment, the barrier, the max-over-ranks timing,
and the whole-job rate of independent replicas (no collective on the data path)."""
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


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import bench

    w, r, loc = bench.dist_setup()
    cpu = torch.device("cpu")
    bench.barrier(w, cpu)
    t_max = bench.max_over_ranks(w, 10.0 + 5.0 * r, cpu)  # rank r "took" 10 + 5r ms
    rate = bench.whole_job_rate(w, 1e12, t_max)
    bench.barrier(w, cpu)
    q.put((r, w, loc, dist.get_backend(), t_max, rate))
    dist.destroy_process_group()


def test_two_rank_gloo_timing_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[0] for x in res] == [0, 1]
    for r, w, loc, backend, t_max, rate in res:
        assert w == 2 and loc == r and backend == "gloo"
        assert t_max == 15.0  # the slowest rank sets the time
        assert rate == pytest.approx(2 * 1e12 / 15e-3)  # both ranks' units over the slowest time


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(1, 3.5, None) == 3.5
    assert bench.whole_job_rate(1, 10.0, 2.0) == pytest.approx(5000.0)
