"""Expert-parallel split on CPU: two and three gloo ranks, each serving the
experts `expert_range` gives it (rank 0 also the shared expert), reduce their
partial outputs with one all_reduce(SUM); the sum is the whole step.  The
partials come from the oracle, so this covers the host side of the split (the
partition and the reduction); the GPU tests cover each rank's launch."""
import multiprocessing as mp
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case():
    from quantized_moe_routed_gb300.inputs import Workload, make_inputs, make_shared_weights
    wl = Workload("ep", T=5, H=128, I=64, E=11, k=3, routing="uniform", seed=71)
    x, ids, w, W = make_inputs(wl, experts="all")
    return wl, x, ids, w, W, make_shared_weights(wl)


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from quantized_moe_routed_gb300 import expert_range
        from quantized_moe_routed_gb300.inputs import expert_slice
        wl, x, ids, w, W, S = _case()
        lo, hi = expert_range(wl.E, rank, world)
        y, bad = oracle.moe_forward(x, ids, w, expert_slice(W, lo, hi), e_range=(lo, hi), E=wl.E,
                                    shared=S if rank == 0 else None)
        t = torch.from_numpy(y)
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        q.put((rank, lo, hi, bad, t.numpy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_ranks_partial_outputs_sum_to_the_whole_step(world):
    sys.path.insert(0, ROOT)
    import oracle
    wl, x, ids, w, W, S = _case()
    y_full, _ = oracle.moe_forward(x, ids, w, W, shared=S)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted((q.get(timeout=180) for _ in procs), key=lambda o: o[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out][0] == 0 and out[-1][2] == wl.E
    assert all(out[i][2] == out[i + 1][1] for i in range(world - 1))      # contiguous, disjoint
    for _, lo, hi, bad, y in out:
        assert bad == 0                                                  # other ranks' ids are not errors
        assert np.allclose(y, y_full, rtol=1e-12, atol=1e-14 * np.abs(y_full).max())


def test_expert_range_partition():
    sys.path.insert(0, ROOT)
    from quantized_moe_routed_gb300 import MoeError, expert_range
    for E in (1, 7, 16, 256):
        for world in range(1, min(E, 9) + 1):
            rs = [expert_range(E, r, world) for r in range(world)]
            assert rs[0][0] == 0 and rs[-1][1] == E
            assert all(a[1] == b[0] for a, b in zip(rs, rs[1:]))
            sizes = [hi - lo for lo, hi in rs]
            assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 1
    for bad in ((4, 0, 5), (4, 4, 2), (4, -1, 2), (8, 0, 0)):
        with pytest.raises(MoeError):
            expert_range(*bad)
