"""GPU parity of the shared expert (one always-on expert added with weight 1
after the routed slots, inside the same launch) and of expert ranges (a plan
serving experts [e_lo, e_hi) of E, its partial y summed with the other
ranges' outside the library) against the oracle, through the C ABI, on every
kernel: the small-launch tensor-core kernel (one token), the tensor-core
ticket kernel (24 tokens), the register kernel, and a prefill launch.
Tolerance: max|y - y_ref| / max|y_ref| <= 2e-3."""
import numpy as np
import pytest
import torch

import oracle
from quantized_moe_routed_gb300 import MoePlan, binding
from quantized_moe_routed_gb300.inputs import (WORKLOADS, Workload, expert_slice, make_expert_weights,
                                               make_shared_weights, make_topk_ids, make_topk_w, make_x,
                                               touched_experts)

pytestmark = pytest.mark.gpu
TOL = 2e-3
DEV = "cuda:0"
KERNELS = {"auto": binding.MOE_KERNEL_AUTO, "register": binding.MOE_KERNEL_REGISTER,
           "tensor": binding.MOE_KERNEL_TENSOR}
SHAPES = {"decode": WORKLOADS["decode"], "upper_decode": WORKLOADS["upper_decode"],
          "t40": Workload("t40", T=40, H=1024, I=512, E=32, k=8, routing="uniform", seed=61),
          "t3": Workload("t3", T=3, H=512, I=768, E=16, k=4, routing="uniform", seed=62)}


def rel_err(y, y_ref):
    y = np.asarray(y, dtype=np.float64)
    den = np.abs(y_ref).max()
    if not np.all(np.isfinite(y)):
        return np.inf
    return float(np.abs(y - y_ref).max() / den)


def cpu(W, experts):
    out = {}
    for k, v in W.items():
        c = torch.zeros(v.shape, dtype=v.dtype)
        for e in experts:
            c[e] = v[e].cpu()
        out[k] = c
    return out


@pytest.fixture(scope="module")
def cache():
    return {}


def case(name, cache):
    if name not in cache:
        wl = SHAPES[name]
        x, ids, w = make_x(wl), make_topk_ids(wl), make_topk_w(wl)
        used = touched_experts(ids, wl.E)
        W = make_expert_weights(wl, device=DEV, experts=used, fill="random")
        S = make_shared_weights(wl, device=DEV)
        Sc = {k: v.cpu() for k, v in S.items()}
        Wc = cpu(W, used)
        y_ref, bad = oracle.moe_forward(x, ids, w, Wc, shared=Sc)
        assert bad == 0
        cache[name] = (wl, x, ids, w, W, S, Wc, Sc, y_ref)
    return cache[name]


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("name", list(SHAPES))
def test_shared_expert_parity(name, kernel, cache):
    wl, x, ids, w, W, S, Wc, Sc, y_ref = case(name, cache)
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=wl.T, strict=False, kernel=KERNELS[kernel], shared=S)
    ws = plan.new_workspace()
    xd, idd, wd = x.to(DEV), ids.to(DEV), w.to(DEV)
    y = plan.step(xd, idd, wd, ws)
    assert plan.check(ws) == 0
    err = rel_err(y.cpu().numpy(), y_ref)
    print(f"{name} {kernel}: shared expert, rel err {err:.3e}, stats {plan.stats()}")
    assert err <= TOL
    y2 = plan.step(xd, idd, wd, ws)                       # bitwise reproducible
    assert plan.check(ws) == 0 and torch.equal(y, y2)
    if kernel == "register":
        assert plan.stats()["tensor_launches"] == 0


def test_shared_expert_alone_with_every_slot_empty(cache):
    wl, x, ids, w, W, S, Wc, Sc, _ = case("t3", cache)
    empty = torch.full_like(ids, -1)
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=wl.T, shared=S)
    ws = plan.new_workspace()
    y = plan.step(x.to(DEV), empty.to(DEV), w.to(DEV), ws)
    assert plan.check(ws) == 0
    y_ref, _ = oracle.moe_forward(x, empty, w, Wc, shared=Sc)
    assert rel_err(y.cpu().numpy(), y_ref) <= TOL


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("name,cut", [("decode", 128), ("upper_decode", 100), ("t40", 9), ("t3", 5)])
def test_expert_ranges_sum_to_the_whole_step(name, cut, kernel, cache):
    """Two plans over [0, cut) (with the shared expert) and [cut, E), each
    holding only its experts' arrays: their outputs sum to the whole step."""
    wl, x, ids, w, W, S, Wc, Sc, y_ref = case(name, cache)
    xd, idd, wd = x.to(DEV), ids.to(DEV), w.to(DEV)
    ys = []
    for (lo, hi), sh in (((0, cut), S), ((cut, wl.E), None)):
        plan = MoePlan(expert_slice(W, lo, hi), wl.H, wl.I, wl.E, wl.k, T_max=wl.T, strict=False,
                       kernel=KERNELS[kernel], shared=sh, e_range=(lo, hi))
        ws = plan.new_workspace()
        y = plan.step(xd, idd, wd, ws)
        assert plan.check(ws) == 0                        # the other range's ids are not errors
        ya, _ = oracle.moe_forward(x, ids, w, {k: v[lo:hi].contiguous() for k, v in Wc.items()},
                                   e_range=(lo, hi), E=wl.E, shared=None if sh is None else Sc)
        assert rel_err(y.cpu().numpy(), ya) <= TOL * np.abs(y_ref).max() / max(np.abs(ya).max(), 1e-30) + TOL
        ys.append(y.cpu().numpy().astype(np.float64))
    err = rel_err(ys[0] + ys[1], y_ref)
    print(f"{name} {kernel}: ranges [0,{cut}) + [{cut},{wl.E}): rel err {err:.3e}")
    assert err <= TOL


def test_expert_range_flags_only_ids_past_E(cache):
    wl, x, ids, w, W, S, Wc, Sc, _ = case("t3", cache)
    bad = ids.clone()
    bad[0, 1] = wl.E + 3
    plan = MoePlan(expert_slice(W, 0, 8), wl.H, wl.I, wl.E, wl.k, T_max=wl.T, e_range=(0, 8))
    ws = plan.new_workspace()
    plan.step(x.to(DEV), bad.to(DEV), w.to(DEV), ws)
    assert plan.check(ws) == binding.MOE_ERR_BAD_EXPERT_ID


def test_plan_refuses_bad_ranges_and_partial_shared_sets(cache):
    wl, x, ids, w, W, S, Wc, Sc, _ = case("t3", cache)
    for rng in ((4, 4), (-1, 3), (3, wl.E + 1)):
        with pytest.raises(binding.MoeError) as ei:
            MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=wl.T, e_range=rng)
        assert ei.value.status == binding.MOE_ERR_INVALID_ARG
    with pytest.raises(binding.MoeError):
        MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=wl.T, shared={**S, "ts": torch.ones(2, device=DEV)})
