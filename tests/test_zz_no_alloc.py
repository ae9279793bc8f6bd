"""moe_decode_static (the decode step on the library's own per-device scratch)
against moe_decode with a caller workspace: two calls in a row on the same
inputs.  moe_decode_static always runs the register kernel, so the reference
is moe_decode on a plan that also takes the register kernel: the two must be
bitwise equal (same kernel, same inputs, a deterministic combine); both are
also held to the oracle's 2e-3 tolerance.  Named to be collected last, so it
runs both after the other GPU tests and alone."""
import numpy as np
import pytest
import torch

import oracle
from quantized_moe_routed_gb300 import MoeError, MoePlan, binding
from quantized_moe_routed_gb300.inputs import (WORKLOADS, make_expert_weights, make_topk_ids, make_topk_w, make_x,
                                               touched_experts)

pytestmark = pytest.mark.gpu
TOL = 2e-3
DEV = "cuda:0"


def rel_err(y, y_ref):
    y, y_ref = np.asarray(y, np.float64), np.asarray(y_ref, np.float64)
    den = np.abs(y_ref).max()
    return 0.0 if den == 0 and np.all(y == 0) else float(np.abs(y - y_ref).max() / den)


@pytest.mark.parametrize("name", ["decode", "upper_decode"])
def test_static_scratch_matches_workspace_path(name):
    wl = WORKLOADS[name]
    x, ids, w = make_x(wl), make_topk_ids(wl), make_topk_w(wl)
    used = touched_experts(ids, wl.E)
    W = make_expert_weights(wl, device=DEV, experts=used, fill="random")
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=wl.T, strict=True, kernel=binding.MOE_KERNEL_REGISTER)
    ws = plan.new_workspace()
    xd, idd, wd = x.to(DEV), ids.to(DEV), w.to(DEV)
    y_ws = plan.step(xd, idd, wd, ws)
    assert plan.check(ws) == 0
    assert plan.stats()["tensor_launches"] == 0
    Wc = {}
    for kk, v in W.items():
        c = torch.zeros(v.shape, dtype=v.dtype)
        for e in used:
            c[e] = v[e].cpu()
        Wc[kk] = c
    y_ref, _ = oracle.moe_forward(x, ids, w, Wc)
    assert rel_err(y_ws.cpu().numpy(), y_ref) <= TOL
    for call in range(2):
        y = torch.full((wl.T, wl.H), float("nan"), dtype=torch.float32, device=DEV)
        binding.moe_decode_static(plan.handle, xd, idd, wd, y, check=True)
        err = rel_err(y.cpu().numpy(), y_ref)
        print(f"{name}: call {call}: rel err vs oracle {err:.3e}")
        assert torch.equal(y, y_ws), f"call {call}: static scratch differs from the workspace path"
        assert err <= TOL


def test_static_scratch_refuses_what_does_not_fit():
    # T above the decode bound
    wl = WORKLOADS["tiny"]
    W = make_expert_weights(wl, device=DEV, experts=range(wl.E), fill="random")
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=64, strict=True)
    z = dict(dtype=torch.float32, device=DEV)
    with pytest.raises(MoeError) as ei:
        binding.moe_decode_static(plan.handle, torch.zeros((25, wl.H), dtype=torch.bfloat16, device=DEV),
                                  torch.zeros((25, wl.k), dtype=torch.int32, device=DEV),
                                  torch.zeros((25, wl.k), **z), torch.empty((25, wl.H), **z))
    assert ei.value.status == binding.MOE_ERR_INVALID_ARG
    # a shape whose per-pair outputs alone exceed the 16 MiB scratch
    # (24 tokens x 16 slots x 16384 floats); refused before any launch
    H, I, E, k, T = 16384, 128, 16, 16, 24
    u8 = dict(dtype=torch.uint8, device=DEV)
    Wb = {"gate_q": torch.zeros((E, I, H // 2), **u8), "up_q": torch.zeros((E, I, H // 2), **u8),
          "down_q": torch.zeros((E, H, I // 2), **u8), "gate_s": torch.zeros((E, I, H // 16), **u8),
          "up_s": torch.zeros((E, I, H // 16), **u8), "down_s": torch.zeros((E, H, I // 16), **u8),
          "gate_ts": torch.ones((E,), **z), "up_ts": torch.ones((E,), **z), "down_ts": torch.ones((E,), **z)}
    big = MoePlan(Wb, H, I, E, k, T_max=T, strict=True)
    with pytest.raises(MoeError) as ei:
        binding.moe_decode_static(big.handle, torch.zeros((T, H), dtype=torch.bfloat16, device=DEV),
                                  torch.zeros((T, k), dtype=torch.int32, device=DEV), torch.zeros((T, k), **z),
                                  torch.empty((T, H), **z))
    assert ei.value.status == binding.MOE_ERR_UNSUPPORTED_SHAPE
    # the small case still runs after the refusals
    x, ids, w = make_x(wl).to(DEV), make_topk_ids(wl).to(DEV), make_topk_w(wl).to(DEV)
    y = torch.empty((wl.T, wl.H), **z)
    binding.moe_decode_static(plan.handle, x, ids, w, y, check=True)
    assert torch.isfinite(y).all()
