"""Host-side argument checks of the Python binding that need no GPU: a call
whose buffers disagree with the plan's shape is refused before anything is
queued (the routing kernel writes T*top_k ids and weights, so a narrower
buffer would take an out-of-bounds device write)."""
import pytest
import torch

from quantized_moe_routed_gb300 import MoeError, MoePlan, binding


def _host_plan(E=16, k=4, H=256):
    """A MoePlan shell with CPU tensors standing in for the weights: enough
    for the binding's checks, which run before any library call."""
    plan = MoePlan.__new__(MoePlan)
    plan.weights = {"gate_q": torch.zeros(1, dtype=torch.uint8)}
    plan.H, plan.I, plan.E, plan.top_k, plan.T_max = H, 128, E, k, 8
    plan.handle = None
    return plan


@pytest.mark.parametrize("ids_shape,w_shape", [((4, 2), None), (None, (4, 3)), ((3, 4), (3, 4)), ((4, 4, 1), None)])
def test_route_refuses_outputs_that_are_not_T_by_top_k(ids_shape, w_shape):
    plan = _host_plan()
    lg = torch.zeros((4, 16), dtype=torch.float32)
    ids = None if ids_shape is None else torch.empty(ids_shape, dtype=torch.int32)
    w = None if w_shape is None else torch.empty(w_shape, dtype=torch.float32)
    with pytest.raises(MoeError) as ei:
        plan.route(lg, ids=ids, w=w)
    assert ei.value.status == binding.MOE_ERR_INVALID_ARG


def test_route_refuses_logits_of_the_wrong_width():
    plan = _host_plan()
    with pytest.raises(MoeError) as ei:
        plan.route(torch.zeros((4, 8), dtype=torch.float32))
    assert ei.value.status == binding.MOE_ERR_INVALID_ARG


def test_route_refuses_logits_on_another_device():
    plan = _host_plan()
    plan.weights = {"gate_q": torch.zeros(1, dtype=torch.uint8, device="meta")}
    with pytest.raises(MoeError) as ei:
        plan.route(torch.zeros((4, 16), dtype=torch.float32))
    assert ei.value.status == binding.MOE_ERR_INVALID_ARG


def test_step_refuses_ids_of_the_wrong_width():
    plan = _host_plan()
    x = torch.zeros((2, 256), dtype=torch.bfloat16)
    with pytest.raises(MoeError) as ei:
        plan.step(x, torch.zeros((2, 3), dtype=torch.int32), torch.zeros((2, 3)), ws=None)
    assert ei.value.status == binding.MOE_ERR_INVALID_ARG
