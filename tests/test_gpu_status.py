"""Device and host statuses on the GPU, through the C ABI:

* MOE_ERR_SCALE: a weight block scale with its sign bit set, or the NaN code
  0x7F, in a plan that may run the tensor-core kernels (the block-scaled MMA
  reads E4M3 scales as unsigned): moe_workspace_init scans every weight scale,
  so it is reported even for an expert no token routes to; the register and
  row kernels decode the sign and give the oracle's y for the same weights.
* MOE_ERR_RANGE: tensor scales large enough that h overflows fp32, on every
  kernel.
* Workspace ownership: a launch on a workspace that is still in flight on
  another stream is ordered after it (its stream waits on the library's event),
  so the two never overlap; another workspace runs at once.  The first stream
  is held back by a timed sleep kernel queued ahead of its step (a bounded
  delay, not a wait on anything).  MOE_ERR_WORKSPACE_BUSY, a second thread
  claiming the workspace from another stream between another thread's claim
  and its event record, is a window of microseconds and not tested here."""
import numpy as np
import pytest
import torch

import oracle
from quantized_moe_routed_gb300 import MoePlan, binding
from quantized_moe_routed_gb300.inputs import (Workload, make_expert_weights, make_topk_ids, make_topk_w, make_x,
                                               touched_experts)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = 2e-3
SLEEP_CYCLES = 200_000_000  # about 0.1 s at 2 GHz


def rel_err(y, y_ref):
    y = np.asarray(y, dtype=np.float64)
    if not np.all(np.isfinite(y)):
        return np.inf
    return float(np.abs(y - y_ref).max() / max(np.abs(y_ref).max(), 1e-30))


def case(T, H=1024, I=512, E=16, k=4, seed=131):
    wl = Workload("status", T=T, H=H, I=I, E=E, k=k, routing="uniform", seed=seed)
    x, ids, w = make_x(wl), make_topk_ids(wl), make_topk_w(wl)
    used = touched_experts(ids, wl.E)
    W = make_expert_weights(wl, device=DEV, experts=used, fill="zero")
    return wl, x, ids, w, W, used


def run(wl, x, ids, w, W, **kw):
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=wl.T, **kw)
    ws = plan.new_workspace()
    y = plan.step(x.to(DEV), ids.to(DEV), w.to(DEV), ws)
    return plan, ws, y, plan.check(ws)


def poke_scale(W, used, name, code, mode="set"):
    """One block-scale byte of the first used expert: its sign bit set
    (mode "sign") or replaced by `code` (mode "set")."""
    e = int(used[0])
    s = W[name]
    v = int(s[e, 3, 5].item())
    s[e, 3, 5] = (v | 0x80) if mode == "sign" else code


@pytest.mark.parametrize("T,kernel", [(40, binding.MOE_KERNEL_TENSOR), (2, binding.MOE_KERNEL_AUTO)])
@pytest.mark.parametrize("name,mode,code", [("gate_s", "sign", 0), ("down_s", "sign", 0), ("up_s", "set", 0x7F)])
def test_tensor_kernels_report_an_unreadable_scale(T, kernel, name, mode, code):
    wl, x, ids, w, W, used = case(T)
    poke_scale(W, used, name, code, mode)
    plan, ws, y, st = run(wl, x, ids, w, W, kernel=kernel)
    s = plan.stats()
    assert s["tensor_launches"] == 1
    if T == 2:
        assert s["small_launches"] == 1
    assert st == binding.MOE_ERR_SCALE, binding.STATUS_NAMES.get(st)
    # cleared by moe_check; a clean plan on the same workspace reports nothing
    assert plan.check(ws) == 0


def test_unreadable_scale_of_an_unrouted_expert_is_reported():
    """The scan reads every expert's scales, not only the routed ones'."""
    wl, x, ids, w, W, used = case(40, E=256)
    unused = [e for e in range(wl.E) if e not in set(int(u) for u in used)]
    assert unused
    W["down_s"][unused[0], 0, 0] = 0x7F
    plan, ws, y, st = run(wl, x, ids, w, W, kernel=binding.MOE_KERNEL_TENSOR)
    assert st == binding.MOE_ERR_SCALE


def test_tensor_kernels_clean_scales_report_nothing():
    for T, kernel in ((40, binding.MOE_KERNEL_TENSOR), (2, binding.MOE_KERNEL_AUTO)):
        wl, x, ids, w, W, used = case(T)
        plan, ws, y, st = run(wl, x, ids, w, W, kernel=kernel)
        assert st == 0 and plan.stats()["tensor_launches"] == 1


@pytest.mark.parametrize("T,kernel,counter", [(1, binding.MOE_KERNEL_AUTO, "gemv_launches"),
                                              (3, binding.MOE_KERNEL_REGISTER, "decode_launches")])
def test_register_and_row_kernels_decode_a_negative_scale(T, kernel, counter):
    """The same negative scale is a legal E4M3 value for the kernels that
    decode it: y matches the oracle, which decodes the sign too."""
    wl, x, ids, w, W, used = case(T, H=2048)
    poke_scale(W, used, "gate_s", 0, "sign")
    poke_scale(W, used, "down_s", 0, "sign")
    plan, ws, y, st = run(wl, x, ids, w, W, kernel=kernel)
    assert st == 0 and plan.stats()[counter] >= 1 and plan.stats()["tensor_launches"] == 0
    Wc = {n: v.cpu() for n, v in W.items()}
    y_ref, _ = oracle.moe_forward(x, ids, w, Wc)
    assert rel_err(y.cpu().numpy(), y_ref) <= TOL


@pytest.mark.parametrize("T,kernel,counter", [(1, binding.MOE_KERNEL_AUTO, "gemv_launches"),
                                              (3, binding.MOE_KERNEL_REGISTER, "decode_launches"),
                                              (2, binding.MOE_KERNEL_AUTO, "small_launches"),
                                              (40, binding.MOE_KERNEL_TENSOR, "tensor_launches")])
def test_h_overflow_reports_range(T, kernel, counter):
    """Gate and up tensor scales of 1e30 put SiLU(g) * u near 1e60 for some
    rows of I: not finite in fp32, reported as MOE_ERR_RANGE."""
    wl, x, ids, w, W, used = case(T, H=2048)
    for e in used:
        W["gate_ts"][int(e)] = 1e30
        W["up_ts"][int(e)] = 1e30
    plan, ws, y, st = run(wl, x, ids, w, W, kernel=kernel)
    assert plan.stats()[counter] >= 1
    assert st == binding.MOE_ERR_RANGE, binding.STATUS_NAMES.get(st)


def _ordered(first, second):
    """True when event `second` completed after event `first` (both done)."""
    return first.elapsed_time(second) >= 0.0


def test_workspace_in_flight_on_another_stream_is_ordered():
    wl, x, ids, w, W, used = case(2, H=2048)
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=wl.T)
    xd, idd, wd = x.to(DEV), ids.to(DEV), w.to(DEV)
    a, b = torch.cuda.Stream(), torch.cuda.Stream()
    ws = plan.new_workspace()
    ws2 = plan.new_workspace()
    torch.cuda.synchronize()
    ya = torch.empty(wl.T, wl.H, dtype=torch.float32, device=DEV)
    yb = torch.empty_like(ya)
    yc = torch.empty_like(ya)
    ev = {n: torch.cuda.Event(enable_timing=True) for n in ("a", "b", "c")}
    with torch.cuda.stream(a):
        torch.cuda._sleep(SLEEP_CYCLES)
    binding.moe_decode(plan.handle, xd, idd, wd, ya, ws, a)
    ev["a"].record(a)
    # the same workspace from stream b, while a's step is queued behind the sleep:
    # accepted, and b's step runs after a's
    binding.moe_decode(plan.handle, xd, idd, wd, yb, ws, b)
    ev["b"].record(b)
    # another workspace: no ordering with a
    c = torch.cuda.Stream()
    binding.moe_decode(plan.handle, xd, idd, wd, yc, ws2, c)
    ev["c"].record(c)
    torch.cuda.synchronize()
    assert _ordered(ev["a"], ev["b"])
    assert not _ordered(ev["a"], ev["c"])  # c did not wait for the sleep
    assert plan.check(ws, b) == 0 and plan.check(ws2, c) == 0
    assert torch.equal(ya, yb) and torch.equal(ya, yc)
    Wc = {n: v.cpu() for n, v in W.items()}
    y_ref, _ = oracle.moe_forward(x, ids, w, Wc)
    assert rel_err(yb.cpu().numpy(), y_ref) <= TOL


def test_static_scratch_in_flight_on_another_stream_is_ordered():
    wl, x, ids, w, W, used = case(2, H=2048)
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=wl.T)
    xd, idd, wd = x.to(DEV), ids.to(DEV), w.to(DEV)
    a, b = torch.cuda.Stream(), torch.cuda.Stream()
    ya = torch.empty(wl.T, wl.H, dtype=torch.float32, device=DEV)
    yb = torch.empty_like(ya)
    binding.moe_decode_static(plan.handle, xd, idd, wd, ya, stream=a)  # first call: set-up
    a.synchronize()
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(a):
        torch.cuda._sleep(SLEEP_CYCLES)
    binding.moe_decode_static(plan.handle, xd, idd, wd, ya, stream=a)
    ea.record(a)
    binding.moe_decode_static(plan.handle, xd, idd, wd, yb, stream=b)
    eb.record(b)
    torch.cuda.synchronize()
    assert _ordered(ea, eb)
    assert torch.equal(ya, yb)
