"""GPU parity of the top-k routing kernel (moe_route) against the oracle, and
of the routed step (routing, then the step, on one stream) against the
oracle's routing followed by its step.  Expert ids are compared bit-exactly
(both sides select by exact comparisons of the same fp32 logits).  The weights
agree within 4e-6 relative: the kernel's expf (<= 2 ulp), the fp32 difference
of two logits of magnitude <= 6 (<= 3.6e-7), a sequential fp32 sum of up to
16 terms (<= 15 x 2^-24) and the division add up to about 1.6e-6 against the
oracle's double arithmetic rounded once.  The routed step's y stays within
the step's 2e-3 tolerance."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from quantized_moe_routed_gb300 import MoeError, MoePlan, binding
from quantized_moe_routed_gb300.inputs import Workload, make_expert_weights, make_router_logits, make_x

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _plan(T, E, k, H=256, I=128, full=False):
    """A plan of E experts; routing reads no weights, so unless `full` only
    expert 0 is drawn and the rest are zero."""
    wl = Workload("route", T=T, H=H, I=I, E=E, k=k, routing="uniform", seed=31)
    W = make_expert_weights(wl, device=DEV, experts=None if full else [0], fill="zero")
    return wl, W, MoePlan(W, H, I, E, k, T_max=max(T, 1))


def _check(ids, w, logits, k):
    ref_ids, ref_w = oracle.route(logits, k)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    wg = w.cpu().numpy()
    assert np.all(np.abs(wg - ref_w) <= 4e-6 * np.abs(ref_w) + 1e-37)


@pytest.mark.parametrize("T,E,k", [(1, 256, 8), (16, 256, 8), (24, 256, 8), (5, 7, 7), (3, 1024, 16),
                                   (40, 33, 4), (9, 64, 1)])
def test_route_matches_oracle(T, E, k):
    wl, W, plan = _plan(T, E, k)
    logits = make_router_logits(wl)
    ids, w = plan.route(logits.to(DEV))
    torch.cuda.synchronize()
    _check(ids, w, logits, k)
    assert plan.stats()["route_launches"] == 1


def test_route_ties_nan_and_extremes():
    lg = np.array([[0.5, 2.0, 2.0, -1.0, np.nan, 3.0],
                   [1.0, 1.0, 1.0, 1.0, 1.0, 1.0],
                   [1000.0, 999.0, -1000.0, 998.0, 0.0, 0.0],
                   [-np.inf] * 6,
                   [np.nan, -5.0, 0.25, np.nan, 0.5, -5.0],
                   [1.0, np.inf, 0.0, np.inf, 5.0, np.inf],
                   [np.inf, -np.inf, 3.0, 2.0, 1.0, 0.0]], np.float32)
    wl, W, plan = _plan(7, 6, 3)
    ids, w = plan.route(torch.from_numpy(lg).to(DEV))
    torch.cuda.synchronize()
    assert ids.cpu().tolist() == [[5, 1, 2], [0, 1, 2], [0, 1, 3], [0, 1, 2], [4, 2, 1], [1, 3, 5], [0, 2, 3]]
    assert bool((w[3] == 0).all())
    assert w[6].cpu().tolist() == [1.0, 0.0, 0.0]      # a +inf winner takes the whole weight
    _check(ids, w, lg, 3)


def test_route_refuses_mismatched_outputs():
    """The kernel writes T*top_k ids and weights: narrower caller buffers are
    refused on the host, before any launch."""
    wl, W, plan = _plan(4, 16, 4)
    lg = torch.zeros((4, 16), dtype=torch.float32, device=DEV)
    for ids, w in ((torch.empty((4, 2), dtype=torch.int32, device=DEV), None),
                   (None, torch.empty((4, 3), dtype=torch.float32, device=DEV)),
                   (torch.empty((3, 4), dtype=torch.int32, device=DEV), torch.empty((3, 4), device=DEV))):
        with pytest.raises(MoeError) as ei:
            plan.route(lg, ids=ids, w=w)
        assert ei.value.status == binding.MOE_ERR_INVALID_ARG
    with pytest.raises(MoeError):
        plan.route(torch.zeros((4, 8), dtype=torch.float32, device=DEV))    # not [T, E]
    assert plan.stats()["route_launches"] == 0


def test_route_is_bitwise_reproducible():
    wl, W, plan = _plan(24, 256, 8)
    logits = make_router_logits(wl).to(DEV)
    a = plan.route(logits)
    b = plan.route(logits)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("T,k", [(1, 8), (12, 4)])
def test_routed_step_matches_the_oracle_chain(T, k):
    """Routing then the step on one stream (the register kernel at one token,
    the tensor-core kernel at twelve) against oracle routing then the oracle
    step."""
    wl, W, plan = _plan(T, 16, k, H=512, I=256, full=True)
    ws = plan.new_workspace()
    x, logits = make_x(wl), make_router_logits(wl)
    y = plan.step_logits(x.to(DEV), logits.to(DEV), ws)
    assert plan.check(ws) == 0
    ref_ids, ref_w = oracle.route(logits, k)
    y_ref, bad = oracle.moe_forward(x, torch.from_numpy(ref_ids), torch.from_numpy(ref_w),
                                    {n: v.cpu() for n, v in W.items()})
    assert bad == 0
    err = float(np.abs(y.cpu().numpy() - y_ref).max() / np.abs(y_ref).max())
    assert err <= 2e-3, err


def test_route_rejections():
    wl, W, plan = _plan(2, 4, 8)                       # top_k > E: no routing
    lg = torch.zeros((2, 4), dtype=torch.float32, device=DEV)
    with pytest.raises(MoeError) as ei:
        plan.route(lg)
    assert ei.value.status == binding.MOE_ERR_UNSUPPORTED_SHAPE
    wl, W, plan = _plan(2, 8, 2)
    with pytest.raises(MoeError) as ei:                # T > T_max
        plan.route(torch.zeros((3, 8), dtype=torch.float32, device=DEV))
    assert ei.value.status == binding.MOE_ERR_INVALID_ARG
    buf = torch.zeros(2 * 8 + 1, dtype=torch.float32, device=DEV)
    ids = torch.empty((2, 2), dtype=torch.int32, device=DEV)
    w = torch.empty((2, 2), dtype=torch.float32, device=DEV)
    lib = binding.load_library()
    P = binding._ptr
    mis = ctypes.c_void_p(buf.data_ptr() + 2)          # 2-byte offset: misaligned
    assert lib.moe_route(plan.handle, mis, 2, P(ids), P(w), None) == binding.MOE_ERR_MISALIGNED
    assert lib.moe_route(plan.handle, None, 0, None, None, None) == binding.MOE_OK     # T == 0
    assert plan.stats()["route_launches"] == 0
