"""GPU parity of the one-token row kernel (moe_gemv.cu: whole gate/up rows per
CTA, one grid-wide barrier, whole output rows per CTA) against the oracle,
through the C ABI: shapes across its range (H a multiple of 2048, I from 256
to 4096, top-k 1 .. 16), repeated, empty and out-of-range slots, the shared
expert and expert ranges, bitwise reproducibility over consecutive launches
on one workspace (the barrier's count carries over), and the timeout path.
Tolerance: max|y - y_ref| / max|y_ref| <= 2e-3."""
import os

import numpy as np
import pytest
import torch

import oracle
from quantized_moe_routed_gb300 import MoePlan, binding
from quantized_moe_routed_gb300.inputs import (Workload, expert_slice, make_expert_weights, make_shared_weights,
                                               make_topk_ids, make_topk_w, make_x, rotate_ids, rotation_delta,
                                               touched_experts)

pytestmark = pytest.mark.gpu
TOL = 2e-3
DEV = "cuda:0"


def rel_err(y, y_ref):
    y = np.asarray(y, dtype=np.float64)
    if not np.all(np.isfinite(y)):
        return np.inf
    return float(np.abs(y - y_ref).max() / max(np.abs(y_ref).max(), 1e-30))


def weights(wl, ids):
    used = touched_experts(ids, wl.E)
    W = make_expert_weights(wl, device=DEV, experts=used, fill="random")
    Wc = {}
    for n, v in W.items():
        c = torch.zeros(v.shape, dtype=v.dtype)
        for e in used:
            c[e] = v[e].cpu()
        Wc[n] = c
    return W, Wc


def run(wl, ids=None, x=None, w=None, shared=None, strict=True):
    x = make_x(wl) if x is None else x
    ids = make_topk_ids(wl) if ids is None else ids
    w = make_topk_w(wl) if w is None else w
    W, Wc = weights(wl, ids)
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=1, strict=strict, shared=shared)
    ws = plan.new_workspace()
    y = plan.step(x.to(DEV), ids.to(DEV), w.to(DEV), ws)
    st = plan.check(ws)
    return plan, ws, y, st, x, ids, w, W, Wc


@pytest.mark.parametrize("H,I,E,k", [(4096, 1024, 256, 8), (2048, 256, 16, 1), (2048, 768, 32, 4),
                                     (6144, 512, 64, 16), (2048, 4096, 8, 2), (4096, 2048, 128, 8),
                                     (8192, 256, 12, 6)])
def test_gemv_kernel_shapes(H, I, E, k):
    wl = Workload("gemv", T=1, H=H, I=I, E=E, k=k, routing="uniform", seed=91)
    plan, ws, y, st, x, ids, w, W, Wc = run(wl)
    assert st == 0, binding.STATUS_NAMES.get(st)
    s = plan.stats()
    assert s["gemv_launches"] == 1 and s["small_launches"] == 0 and s["tensor_launches"] == 0
    y_ref, _ = oracle.moe_forward(x, ids, w, Wc)
    err = rel_err(y.cpu().numpy(), y_ref)
    print(f"H={H} I={I} E={E} k={k}: rel err {err:.3e}")
    assert err <= TOL


@pytest.mark.parametrize("H,I,E,k", [(16384, 512, 64, 8), (16384, 4096, 32, 16)])
def test_largest_shapes_match_the_oracle(H, I, E, k):
    """H = 16384 (the row kernel's largest): at I = 512 the row kernel takes the
    step; at I = 4096 with 16 slots its shared memory does not hold the layout,
    and the plan takes another kernel.  Either way y matches the oracle."""
    wl = Workload("gemv-max", T=1, H=H, I=I, E=E, k=k, routing="uniform", seed=98)
    plan, ws, y, st, x, ids, w, W, Wc = run(wl)
    assert st == 0, binding.STATUS_NAMES.get(st)
    s = plan.stats()
    if I == 512:
        assert s["gemv_launches"] == 1
    assert s["decode_launches"] == 1
    y_ref, _ = oracle.moe_forward(x, ids, w, Wc)
    err = rel_err(y.cpu().numpy(), y_ref)
    print(f"H={H} I={I} k={k}: rel err {err:.3e}, row kernel {s['gemv_launches']}")
    assert err <= TOL


def test_gemv_repeated_empty_and_bad_slots():
    """One expert named three times (its h is computed once, weighted per
    slot), empty slots, an id >= E (skipped, flagged)."""
    wl = Workload("gemv-dup", T=1, H=2048, I=512, E=16, k=8, routing="uniform", seed=92)
    ids = torch.tensor([[3, 7, 3, -1, 11, 3, 20, 5]], dtype=torch.int32)
    plan, ws, y, st, x, ids, w, W, Wc = run(wl, ids=ids)
    assert st == binding.MOE_ERR_BAD_EXPERT_ID
    y_ref, bad = oracle.moe_forward(x, ids, w, Wc)
    assert bad == 1
    assert rel_err(y.cpu().numpy(), y_ref) <= TOL


def test_gemv_every_slot_empty_gives_zero():
    wl = Workload("gemv-empty", T=1, H=2048, I=256, E=8, k=4, routing="uniform", seed=93)
    ids = torch.full((1, 4), -1, dtype=torch.int32)
    W = make_expert_weights(wl, device=DEV, experts=[0])
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=1, strict=True)
    ws = plan.new_workspace()
    y = plan.step(make_x(wl).to(DEV), ids.to(DEV), make_topk_w(wl).to(DEV), ws)
    assert plan.check(ws) == 0 and bool((y == 0).all()) and plan.stats()["gemv_launches"] == 1


def test_gemv_shared_expert_and_expert_ranges():
    wl = Workload("gemv-shared", T=1, H=4096, I=1024, E=64, k=8, routing="uniform", seed=94)
    x, ids, w = make_x(wl), make_topk_ids(wl), make_topk_w(wl)
    W, Wc = weights(wl, ids)
    S = make_shared_weights(wl, device=DEV)
    Sc = {n: v.cpu() for n, v in S.items()}
    y_ref, _ = oracle.moe_forward(x, ids, w, Wc, shared=Sc)
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=1, strict=True, shared=S)
    ws = plan.new_workspace()
    y = plan.step(x.to(DEV), ids.to(DEV), w.to(DEV), ws)
    assert plan.check(ws) == 0 and plan.stats()["gemv_launches"] == 1
    assert rel_err(y.cpu().numpy(), y_ref) <= TOL
    ys = []
    for (lo, hi), sh in (((0, 21), S), ((21, wl.E), None)):
        pr = MoePlan(expert_slice(W, lo, hi), wl.H, wl.I, wl.E, wl.k, T_max=1, strict=True, shared=sh,
                     e_range=(lo, hi))
        wsr = pr.new_workspace()
        ys.append(pr.step(x.to(DEV), ids.to(DEV), w.to(DEV), wsr).cpu().numpy().astype(np.float64))
        assert pr.check(wsr) == 0 and pr.stats()["gemv_launches"] == 1
    assert rel_err(ys[0] + ys[1], y_ref) <= TOL


def test_gemv_consecutive_launches_bitwise_and_parity():
    """Sixteen launches on one workspace with relabelled ids (the barrier's
    count carries over from launch to launch); each matches the oracle, and
    repeating the sequence reproduces every bit."""
    wl = Workload("gemv-seq", T=1, H=2048, I=1024, E=64, k=8, routing="uniform", seed=95)
    x, ids, w = make_x(wl), make_topk_ids(wl), make_topk_w(wl)
    W = make_expert_weights(wl, device=DEV, experts=None)
    Wc = {n: v.cpu() for n, v in W.items()}
    delta = rotation_delta(ids, wl.E, window=8)
    idr = [rotate_ids(ids, s, delta, wl.E) for s in range(16)]
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=1, strict=True, pdl=True)
    ws = plan.new_workspace()
    xd, wd = x.to(DEV), w.to(DEV)
    runs = []
    for rep in range(2):
        runs.append([plan.step(xd, r.to(DEV), wd, ws).clone() for r in idr])
        assert plan.check(ws) == 0
    for a, b in zip(*runs):
        assert torch.equal(a, b)
    for r, y in zip(idr[:4], runs[0][:4]):
        y_ref, _ = oracle.moe_forward(x, r, w, Wc)
        assert rel_err(y.cpu().numpy(), y_ref) <= TOL
    assert plan.stats()["gemv_launches"] == 32


def test_gemv_poisoned_workspace_times_out_and_recovers():
    """A poisoned workspace leaves the grid barrier's count off a multiple of
    the grid, so one CTA's barrier never opens: its bounded wait expires, the
    launch returns, moe_check reports the timeout, and after
    moe_workspace_init the plan computes correctly again."""
    os.environ["MOE_WAIT_TIMEOUT_MS"] = "200"
    try:
        wl = Workload("gemv-poison", T=1, H=2048, I=256, E=8, k=4, routing="uniform", seed=96)
        x, ids, w = make_x(wl), make_topk_ids(wl), make_topk_w(wl)
        W = make_expert_weights(wl, device=DEV, experts=None)
        plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=1)
    finally:
        del os.environ["MOE_WAIT_TIMEOUT_MS"]
    ws = plan.new_workspace()
    binding.moe_debug_poison_workspace(plan.handle, ws)
    plan.step(x.to(DEV), ids.to(DEV), w.to(DEV), ws)
    assert plan.check(ws) == binding.MOE_ERR_TIMEOUT
    assert plan.stats()["gemv_launches"] == 1
    binding.moe_workspace_init(plan.handle, ws)
    y = plan.step(x.to(DEV), ids.to(DEV), w.to(DEV), ws)
    assert plan.check(ws) == 0
    y_ref, _ = oracle.moe_forward(x, ids, w, {n: v.cpu() for n, v in W.items()})
    assert rel_err(y.cpu().numpy(), y_ref) <= TOL


def test_gemv_is_left_out_where_it_does_not_apply():
    """act_quant plans, register and tensor-core plans, MOE_GEMV=0 and H not
    a multiple of 2048 take the other kernels."""
    wl = Workload("gemv-off", T=1, H=2048, I=256, E=8, k=4, routing="uniform", seed=97)
    x, ids, w = make_x(wl), make_topk_ids(wl), make_topk_w(wl)
    W = make_expert_weights(wl, device=DEV, experts=None)
    for kw in ({"act_quant": True}, {"kernel": binding.MOE_KERNEL_REGISTER}, {"kernel": binding.MOE_KERNEL_TENSOR}):
        plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=1, **kw)
        ws = plan.new_workspace()
        plan.step(x.to(DEV), ids.to(DEV), w.to(DEV), ws)
        assert plan.check(ws) == 0 and plan.stats()["gemv_launches"] == 0
    os.environ["MOE_GEMV"] = "0"
    try:
        plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=1)
    finally:
        del os.environ["MOE_GEMV"]
    ws = plan.new_workspace()
    plan.step(x.to(DEV), ids.to(DEV), w.to(DEV), ws)
    assert plan.check(ws) == 0 and plan.stats()["gemv_launches"] == 0
