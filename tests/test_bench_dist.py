"""The multi-rank host logic of bench.py on CPU: two gloo ranks (replicas only).

Every rank times its own replica; the job's time is the slowest rank's, and the reported
weight GB/s counts every rank's bytes.  No GPU: the collectives run on gloo.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench
    ctx = bench.DistCtx(backend="gloo")
    ctx.barrier()
    ms = 10.0 * (rank + 1)  # rank 1 is the slow one
    ms_max = ctx.max(ms)
    out[rank] = (ctx.world, ctx.rank, ms_max, bench.whole_job_gbs(1_000_000, ms_max, 100, ctx.world))
    ctx.close()


def test_two_gloo_ranks_take_the_slowest_rank_and_count_all_bytes():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert sorted(res) == [0, 1]
    for rank, (w, r, ms_max, gbs) in res.items():
        assert (w, r) == (world, rank)
        assert ms_max == 20.0
        # 2 ranks x 1 MB per step, 100 steps in 20 ms -> 0.2 ms per step -> 10 GB/s
        assert gbs == pytest.approx(10.0)


def test_single_process_needs_no_process_group():
    import bench
    ctx = bench.DistCtx()
    assert ctx.world == int(os.environ.get("WORLD_SIZE", "1")) or ctx.pg is None
    assert ctx.max(3.5) == 3.5
    assert bench.whole_job_gbs(2_000_000, 1.0, 10, 1) == pytest.approx(20.0)
