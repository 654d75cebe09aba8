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


# ---------------------------------------------------------------- one problem split by heads
def test_head_ranges_cover_every_head_once():
    sys.path.insert(0, ROOT)
    from io_aware_exact_13_gb300.shard import head_range, max_heads

    for H in (1, 2, 3, 7, 8, 16, 32, 33):
        for world in (1, 2, 3, 4, 8, 16):
            count = [0] * H
            prev_end = 0
            for r in range(world):
                h0, h1 = head_range(H, world, r)
                assert h0 == prev_end and h1 >= h0  # contiguous, in rank order
                prev_end = h1
                for h in range(h0, h1):
                    count[h] += 1
                assert h1 - h0 in (H // world, -(-H // world))  # sizes differ by at most one
            assert prev_end == H and count == [1] * H
            assert max_heads(H, world) == -(-H // world)


def _oracle_compute(q, k, v, mask, scale, causal):
    import numpy as np
    import torch

    import oracle

    o, l = oracle.attention(q, k, v, mask=mask, scale=scale, causal=causal)
    return torch.from_numpy(np.asarray(o)), torch.from_numpy(np.asarray(l))


def _shard_worker(rank, world, port, q, B, H, N, d, masked):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import bench
    from io_aware_exact_13_gb300.inputs import make_qkv
    from io_aware_exact_13_gb300.shard import sharded_attention

    w, r, _ = bench.dist_setup()
    # every rank draws the same seeded problem and computes only its heads
    qq, kk, vv, mask = make_qkv(B, H, N, d, "bf16", seed=77, mask_frac=0.1 if masked else 0.0)
    args = [t.double() for t in (qq, kk, vv)]
    m = None if mask is None else mask.double()
    h0, h1, o_s, l_s = sharded_attention(*args, mask=m, scale=0.125, causal=True, gather_result=False,
                                         compute=_oracle_compute)
    out, lse = sharded_attention(*args, mask=m, scale=0.125, causal=True, compute=_oracle_compute)
    q.put((r, w, h0, h1, o_s.numpy(), l_s.numpy(), out.numpy(), lse.numpy()))
    dist.destroy_process_group()


@pytest.mark.parametrize("B,H,N,d,masked", [(1, 5, 67, 64, False), (2, 3, 40, 32, True)])
def test_two_rank_head_partition_equals_one_rank(B, H, N, d, masked):
    """Each of two gloo ranks computes its heads of one problem (with the oracle standing
    in for the device forward); the slices cover every (b, h) once, and the gathered
    O and lse equal the whole problem computed by one process."""
    import numpy as np

    sys.path.insert(0, ROOT)
    import oracle
    from io_aware_exact_13_gb300.inputs import make_qkv

    oracle.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, q, B, H, N, d, masked)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=180) for _ in procs), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    qq, kk, vv, mask = make_qkv(B, H, N, d, "bf16", seed=77, mask_frac=0.1 if masked else 0.0)
    ref_o, ref_l = oracle.attention(qq, kk, vv, mask=mask, scale=0.125, causal=True)
    covered = np.zeros(H, dtype=int)
    for r, w, h0, h1, o_s, l_s, out, lse in res:
        assert w == 2
        covered[h0:h1] += 1
        assert o_s.shape == (B, h1 - h0, N, d) and l_s.shape == (B, h1 - h0, N)
        np.testing.assert_array_equal(o_s, ref_o[:, h0:h1])  # the same rows by the same routine
        np.testing.assert_array_equal(l_s, ref_l[:, h0:h1])
        np.testing.assert_array_equal(out, ref_o)  # every rank holds the assembled result
        np.testing.assert_array_equal(lse, ref_l)
    assert covered.tolist() == [1] * H
