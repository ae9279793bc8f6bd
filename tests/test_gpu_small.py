"""GPU parity of the small-launch tensor-core kernel (launches of at most four
tokens and 32 (token, slot) pairs) against the oracle, through the C ABI:
shapes across the static shares (one or several units per CTA, chunk counts
of I that end on a single 256-element chunk, the largest I), duplicate and
empty slots, experts with more pairs than one down group holds, and bitwise
reproducibility.  Tolerance: max|y - y_ref| / max|y_ref| <= 2e-3."""
import numpy as np
import pytest
import torch

import oracle
from quantized_moe_routed_gb300 import MoePlan, binding
from quantized_moe_routed_gb300.inputs import Workload, make_expert_weights, make_topk_ids, make_topk_w, make_x

pytestmark = pytest.mark.gpu
TOL = 2e-3
DEV = "cuda:0"


def rel_err(y, y_ref):
    y = np.asarray(y, dtype=np.float64)
    den = np.abs(y_ref).max()
    if den == 0:
        return 0.0 if np.all(y == 0) else np.inf
    if not np.all(np.isfinite(y)):
        return np.inf
    return float(np.abs(y - y_ref).max() / den)


def run(wl, ids=None, w=None, x=None, kernel=binding.MOE_KERNEL_AUTO):
    x = make_x(wl) if x is None else x
    ids = make_topk_ids(wl) if ids is None else ids
    w = make_topk_w(wl) if w is None else w
    W = make_expert_weights(wl, device=DEV, experts=None)
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=wl.T, strict=True, kernel=kernel)
    ws = plan.new_workspace()
    y = plan.step(x.to(DEV), ids.to(DEV), w.to(DEV), ws)
    st = plan.check(ws)
    y_ref, _ = oracle.moe_forward(x, ids, w, {k: v.cpu() for k, v in W.items()})
    return plan, ws, y, st, y_ref


@pytest.mark.parametrize("T,H,I,E,k", [(1, 256, 256, 4, 1), (1, 512, 768, 8, 2), (2, 1024, 512, 16, 8),
                                       (3, 768, 1280, 12, 8), (4, 512, 256, 40, 8), (4, 2048, 1024, 64, 8),
                                       (2, 512, 512, 32, 16), (1, 256, 4096, 4, 2), (1, 1024, 2048, 8, 4),
                                       (4, 4096, 256, 24, 4)])
def test_small_kernel_shapes(T, H, I, E, k):
    wl = Workload("small", T=T, H=H, I=I, E=E, k=k, routing="uniform", seed=41)
    plan, ws, y, st, y_ref = run(wl)
    assert st == 0, binding.STATUS_NAMES.get(st)
    s = plan.stats()
    assert s["small_launches"] == 1 and s["tensor_launches"] == 1
    err = rel_err(y.cpu().numpy(), y_ref)
    print(f"T={T} H={H} I={I} E={E} k={k}: rel err {err:.3e}")
    assert err <= TOL


def test_small_kernel_duplicates_empty_and_bad_slots():
    """Slots naming one expert several times (33 pairs would not fit: 4 tokens
    x 8 slots, one expert taking 20 of them -> five down groups of four), empty
    slots (id -1), an id >= E (skipped, flagged), and a token with no valid slot
    (y = 0)."""
    wl = Workload("small-dup", T=4, H=512, I=512, E=16, k=8, routing="uniform", seed=42)
    ids = torch.tensor([[3, 3, 3, 3, 3, 5, -1, 7],
                        [3, 3, 3, 3, 3, 9, 5, 20],
                        [-1, -1, -1, -1, -1, -1, -1, -1],
                        [3, 3, 3, 3, 3, 3, 3, 3]], dtype=torch.int32)
    plan, ws, y, st, y_ref = run(wl, ids=ids)
    assert st == binding.MOE_ERR_BAD_EXPERT_ID
    assert plan.stats()["small_launches"] == 1
    assert bool((y[2] == 0).all())
    assert rel_err(y.cpu().numpy(), y_ref) <= TOL


def test_small_kernel_bitwise_reproducible_and_recovers_after_a_launch():
    wl = Workload("small-rep", T=2, H=2048, I=1024, E=64, k=8, routing="uniform", seed=43)
    x, ids, w = make_x(wl), make_topk_ids(wl), make_topk_w(wl)
    W = make_expert_weights(wl, device=DEV, experts=None)
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=wl.T, strict=True)
    ws = plan.new_workspace()
    xd, idd, wd = x.to(DEV), ids.to(DEV), w.to(DEV)
    ys = [plan.step(xd, idd, wd, ws).clone() for _ in range(3)]
    assert plan.check(ws) == 0
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[1], ys[2])
    # a one-token launch on the same workspace after the two-token ones (the
    # one-token row kernel takes it: H is a multiple of 2048), then two tokens again
    y1 = plan.step(xd[:1].contiguous(), idd[:1].contiguous(), wd[:1].contiguous(), ws)
    assert plan.check(ws) == 0
    y_ref, _ = oracle.moe_forward(x[:1], ids[:1], w[:1], {k: v.cpu() for k, v in W.items()})
    assert rel_err(y1.cpu().numpy(), y_ref) <= TOL
    y2 = plan.step(xd, idd, wd, ws)
    assert plan.check(ws) == 0 and torch.equal(y2, ys[0])
    assert plan.stats()["small_launches"] == 4 and plan.stats()["gemv_launches"] == 1


def test_register_kernel_plan_never_takes_the_small_kernel():
    wl = Workload("small-reg", T=1, H=512, I=512, E=8, k=4, routing="uniform", seed=44)
    plan, ws, y, st, y_ref = run(wl, kernel=binding.MOE_KERNEL_REGISTER)
    assert st == 0 and plan.stats()["small_launches"] == 0 and plan.stats()["tensor_launches"] == 0
    assert rel_err(y.cpu().numpy(), y_ref) <= TOL
