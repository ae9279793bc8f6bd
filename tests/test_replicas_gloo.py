"""The N-GPU bench path on CPU: two gloo ranks, as torchrun would start them.

The step does not shard (every GPU runs an independent replica), so the only
cross-rank work is the timing reduction: the slowest rank's time and the bytes
of all ranks over it.  The reference arm runs on rank 0 alone.
"""
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


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms, gbs = bench.aggregate_ranks(0.030 + 0.010 * rank, 56_647_840, world, "cpu")
        q.put((rank, ms, gbs, bench.dist_env()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_all_bytes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, gbs, env in out:
        assert env == (rank, 2, rank)
        assert ms == pytest.approx(0.040)  # rank 1's 40 us: the max over ranks
        assert gbs == pytest.approx(2 * 56_647_840 / 40e-6 / 1e9)


def test_one_rank_reduces_nothing():
    sys.path.insert(0, ROOT)
    import bench
    ms, gbs = bench.aggregate_ranks(0.030, 56_647_840, 1, "cpu")
    assert ms == 0.030 and gbs == pytest.approx(56_647_840 / 30e-6 / 1e9)


def test_reference_arm_runs_on_rank_0_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    # rank 1 returns before touching any input, device or the oracle
    assert bench.run_reference(None) is None
