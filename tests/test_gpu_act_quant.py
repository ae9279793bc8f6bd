"""GPU parity of the single NVFP4 activation quantisation (act_quant plans):
x and h quantised once to NVFP4 before each projection, on the small-launch
and ticket tensor-core kernels, against the oracle's act_quant mode.

Both sides quantise x from the same bf16 values with the same fp32 steps, so
its codes agree exactly.  h is formed in fp32 by the kernels and in float64
(then rounded to fp32) by the oracle, so an element lying within that
rounding of an E2M1 or E4M3 decision boundary may take the neighbouring code
on either side, and both are correct.  The test finds those elements from
the oracle's h (quantised again with every element moved by +-ETA times its
block's largest |h|; ETA = 3e-5 is about 30 times the kernels' fp32 error)
and lets each of them take, in the kernel's output, either its own code or
the neighbouring one: per token the difference is fitted by those elements'
W_down columns, each coefficient snapped to the nearest allowed change.  What
is left must be within 5e-5 of max|y| (fp32 accumulation of the down
projection)."""
import numpy as np
import pytest
import torch

import oracle
from quantized_moe_routed_gb300 import MoePlan, binding
from quantized_moe_routed_gb300.inputs import (WORKLOADS, Workload, make_expert_weights, make_shared_weights,
                                               make_topk_ids, make_topk_w, make_uneven_expert_weights, make_x,
                                               touched_experts)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
ETA = 3e-5
TOL = 5e-5
SHAPES = {"decode": WORKLOADS["decode"],
          "t3": Workload("t3", T=3, H=512, I=768, E=16, k=4, routing="uniform", seed=81),
          "t24": Workload("t24", T=24, H=1024, I=1024, E=64, k=8, routing="uniform", seed=82),
          "t40": Workload("t40", T=40, H=1024, I=512, E=32, k=8, routing="uniform", seed=83)}
KERNELS = {"auto": binding.MOE_KERNEL_AUTO, "tensor": binding.MOE_KERNEL_TENSOR}


def _cpu(W):
    return {k: v.cpu() for k, v in W.items()}


def _one_expert(S):
    """The shared expert's arrays as a one-expert weight dict."""
    out = {n: S[n][None] for n in ("gate_q", "up_q", "down_q", "gate_s", "up_s", "down_s")}
    for i, n in enumerate(("gate_ts", "up_ts", "down_ts")):
        out[n] = S["ts"][i:i + 1]
    return out


def ambiguous(x, ids, w, Wc, Sc=None):
    """Per token, the h elements whose code the fp32 rounding of h may change:
    a list of (column, allowed changes): column = routing weight x W_down's
    column of that element (float64 [H]); allowed = the element's possible
    changes of value (0 and the one-step changes that moving it by +-ETA
    times its block's largest |h| produces)."""
    T, k = ids.shape
    out = [[] for _ in range(T)]
    pairs = [(t, int(ids[t, j]), Wc, float(w[t, j])) for t in range(T) for j in range(k) if int(ids[t, j]) >= 0]
    if Sc is not None:
        S1 = _one_expert(Sc)
        pairs += [(t, 0, S1, 1.0) for t in range(T)]
    xq = {}
    for t, e, WW, wt in pairs:
        if t not in xq:
            xq[t] = oracle.quant_row_nvfp4(x[t].float().numpy())
        _, _, h, _ = oracle.expert_pair(xq[t], e, WW)
        hf = h.astype(np.float32)
        bm = np.abs(hf.astype(np.float64)).reshape(-1, 16).max(axis=1).repeat(16)
        d = (ETA * bm).astype(np.float32)
        q0 = oracle.quant_row_nvfp4(hf)
        qp, qm = oracle.quant_row_nvfp4(hf + d), oracle.quant_row_nvfp4(hf - d)
        idx = np.nonzero((qp != q0) | (qm != q0))[0]
        if idx.size == 0:
            continue
        Wd = oracle.dequant(WW["down_q"][e], WW["down_s"][e], float(WW["down_ts"][e]))
        for i in idx:
            out[t].append((wt * Wd[:, i], sorted({0.0, qp[i] - q0[i], qm[i] - q0[i]})))
    return out


def check(y, x, ids, w, Wc, Sc=None, label=""):
    """y (kernel) against the oracle: per token, the residual is fitted by the
    ambiguous elements' columns, each coefficient snapped to its nearest
    allowed change; what remains must be within TOL of max|y|."""
    y_ref, bad = oracle.moe_forward(x, ids, w, Wc, shared=Sc, act_quant=True)
    assert bad == 0
    amb = ambiguous(x, ids, w, Wc, Sc)
    y = y.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(y))
    scale = np.abs(y_ref).max()
    rest = np.empty_like(y)
    n_amb = n_flip = 0
    for t in range(y.shape[0]):
        r = y[t] - y_ref[t]
        if amb[t]:
            V = np.stack([c for c, _ in amb[t]], axis=1)
            alpha = np.linalg.lstsq(V, r, rcond=None)[0]
            snap = np.array([min(al, key=lambda v: abs(v - a)) for a, (_, al) in zip(alpha, amb[t])])
            r = r - V @ snap
            n_amb += len(amb[t])
            n_flip += int(np.count_nonzero(snap))
        rest[t] = r
    print(f"{label}: max|dy|/max|y| {np.abs(y - y_ref).max() / scale:.3e}, after the ambiguous codes "
          f"{np.abs(rest).max() / scale:.3e} ({n_amb} ambiguous h elements, {n_flip} taken the other way)")
    assert np.abs(rest).max() <= TOL * scale
    return y_ref


@pytest.fixture(scope="module")
def cache():
    return {}


def case(name, cache):
    if name not in cache:
        wl = SHAPES[name]
        x, ids, w = make_x(wl), make_topk_ids(wl), make_topk_w(wl)
        used = touched_experts(ids, wl.E)
        W = make_expert_weights(wl, device=DEV, experts=used, fill="random")
        Wc = _cpu(W)
        cache[name] = (wl, x, ids, w, W, Wc)
    return cache[name]


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("name", list(SHAPES))
def test_act_quant_parity(name, kernel, cache):
    wl, x, ids, w, W, Wc = case(name, cache)
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=wl.T, kernel=KERNELS[kernel], act_quant=True)
    ws = plan.new_workspace()
    y = plan.step(x.to(DEV), ids.to(DEV), w.to(DEV), ws)
    assert plan.check(ws) == 0
    st = plan.stats()
    assert st["small_launches"] + st["tensor_launches"] >= 1
    y_ref = check(y, x, ids, w, Wc, label=f"{name} {kernel}")
    # the mode is on: the four-digit step differs by far more than the tolerance
    y4, _ = oracle.moe_forward(x, ids, w, Wc)
    assert np.abs(y4 - y_ref).max() > 50 * TOL * np.abs(y_ref).max()


@pytest.mark.parametrize("name", ["t3", "t24"])
def test_act_quant_with_the_shared_expert(name, cache):
    wl, x, ids, w, W, Wc = case(name, cache)
    S = make_shared_weights(wl, device=DEV)
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=wl.T, shared=S, act_quant=True)
    ws = plan.new_workspace()
    y = plan.step(x.to(DEV), ids.to(DEV), w.to(DEV), ws)
    assert plan.check(ws) == 0
    check(y, x, ids, w, Wc, Sc=_cpu(S), label=f"{name} shared")


@pytest.mark.parametrize("T", [2, 24, 40])
def test_act_quant_h_slices_binades_apart(T):
    """h rows [128, 256) lie ~15 binades below the rest but carry y: the
    ticket kernel quantises h per 128-row slice and shifts each slice's block
    scales to the row's prescale; here the shift leaves them subnormal, so
    those blocks must be quantised again from h at the row's prescale."""
    wl = Workload("uneven", T=T, H=1024, I=512, E=8, k=2, routing="uniform", seed=84)
    x, ids, w = make_x(wl), make_topk_ids(wl), make_topk_w(wl)
    Wc = make_uneven_expert_weights(wl, 128, 256, 15)
    W = {k: v.to(DEV) for k, v in Wc.items()}
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=wl.T, act_quant=True)
    ws = plan.new_workspace()
    y = plan.step(x.to(DEV), ids.to(DEV), w.to(DEV), ws)
    assert plan.check(ws) == 0
    check(y, x, ids, w, Wc, label=f"uneven T={T}")


def test_act_quant_refusals(cache):
    wl, x, ids, w, W, Wc = case("t3", cache)
    with pytest.raises(binding.MoeError) as ei:
        MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=wl.T, kernel=binding.MOE_KERNEL_REGISTER, act_quant=True)
    assert ei.value.status == binding.MOE_ERR_UNSUPPORTED_SHAPE
    odd = Workload("odd", T=2, H=384, I=256, E=4, k=2, routing="uniform", seed=85)   # H not a multiple of 256
    Wo = make_expert_weights(odd, device=DEV)
    with pytest.raises(binding.MoeError) as ei:
        MoePlan(Wo, odd.H, odd.I, odd.E, odd.k, T_max=odd.T, act_quant=True)
    assert ei.value.status == binding.MOE_ERR_UNSUPPORTED_SHAPE
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=wl.T, act_quant=True)
    y = torch.empty(wl.T, wl.H, dtype=torch.float32, device=DEV)
    with pytest.raises(binding.MoeError) as ei:
        binding.moe_decode_static(plan.handle, x.to(DEV), ids.to(DEV), w.to(DEV), y)
    assert ei.value.status == binding.MOE_ERR_UNSUPPORTED_SHAPE
