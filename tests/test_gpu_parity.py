"""GPU parity of the sm_103a routed-MoE step against the CPU oracle, through
the C ABI.  Tolerance: max|y - y_ref| / max|y_ref| <= 2e-3 (fp32 output; fp16
mma.sync operands on the register kernel, four FP4 digit rows per activation
row on the tensor-core kernel; fp32 accumulation); grouping bit-exact;
repeated runs bitwise identical."""
import os

import numpy as np
import pytest
import torch

import oracle
from quantized_moe_routed_gb300 import MoeError, MoePlan, binding
from quantized_moe_routed_gb300.inputs import (WORKLOADS, Workload, make_expert_weights, make_topk_ids, make_topk_w,
                                               make_x, quantize_nvfp4, touched_experts)

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


def weights_cpu(W, experts):
    """CPU copy of the weights the oracle needs (other experts zero-filled)."""
    out = {}
    for k, v in W.items():
        c = torch.zeros(v.shape, dtype=v.dtype)
        for e in experts:
            c[e] = v[e].cpu()
        out[k] = c
    return out


def run_case(wl, x, ids, w, W, *, strict=True, T_max=None, pdl=False, kernel=binding.MOE_KERNEL_AUTO):
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=T_max or max(wl.T, 1), strict=strict, pdl=pdl, kernel=kernel)
    ws = plan.new_workspace()
    y = plan.step(x.to(DEV), ids.to(DEV), w.to(DEV), ws)
    st = plan.check(ws)
    return plan, ws, y, st


@pytest.fixture(scope="module")
def cache():
    return {}


def workload_inputs(name, cache):
    if name in cache:
        return cache[name]
    wl = WORKLOADS[name]
    x, ids, w = make_x(wl), make_topk_ids(wl), make_topk_w(wl)
    W = make_expert_weights(wl, device=DEV, experts=touched_experts(ids, wl.E), fill="random")
    cache[name] = (wl, x, ids, w, W)
    return cache[name]


def workload_ref(name, cache):
    """The oracle's y over every token of the workload (computed once per module:
    the prefill chunk's 4096 pairs take about 20 s on the host's cores)."""
    key = name + "/ref"
    if key not in cache:
        wl, x, ids, w, W = workload_inputs(name, cache)
        y_ref, bad = oracle.moe_forward(x, ids, w, weights_cpu(W, touched_experts(ids, wl.E)))
        assert bad == 0
        cache[key] = y_ref
    return cache[key]


# ------------------------------------------------------------------ the five workloads at full size
@pytest.mark.parametrize("kernel", [binding.MOE_KERNEL_AUTO, binding.MOE_KERNEL_REGISTER])
@pytest.mark.parametrize("name", ["tiny", "decode", "spec_verify", "upper_decode", "prefill"])
def test_workload_parity(name, kernel, cache):
    """Every element of y, every token (the prefill chunk's 512 included)."""
    wl, x, ids, w, W = workload_inputs(name, cache)
    plan, ws, y, st = run_case(wl, x, ids, w, W, kernel=kernel)
    assert st == 0, binding.STATUS_NAMES.get(st)
    y_ref = workload_ref(name, cache)
    err = rel_err(y.cpu().numpy(), y_ref)
    print(f"{name}: rel err {err:.3e} over {wl.T} tokens")
    assert err <= TOL
    s = plan.stats()
    assert s["decode_launches" if wl.T <= 24 else "prefill_launches"] >= 1 and s["rejected_calls"] == 0
    if kernel == binding.MOE_KERNEL_REGISTER:
        assert s["tensor_launches"] == 0


# ------------------------------------------------------------------ the tensor-core kernel
@pytest.mark.parametrize("name", ["decode", "spec_verify", "upper_decode", "prefill"])
def test_tensor_kernel_workload_parity(name, cache):
    wl, x, ids, w, W = workload_inputs(name, cache)
    plan, ws, y, st = run_case(wl, x, ids, w, W, kernel=binding.MOE_KERNEL_TENSOR)
    assert st == 0, binding.STATUS_NAMES.get(st)
    err = rel_err(y.cpu().numpy(), workload_ref(name, cache))
    print(f"{name} (tensor-core kernel): rel err {err:.3e}")
    assert err <= TOL
    s = plan.stats()
    assert s["tensor_launches"] >= 1 and s["rejected_calls"] == 0


@pytest.mark.parametrize("kernel", [binding.MOE_KERNEL_AUTO, binding.MOE_KERNEL_REGISTER])
def test_prefill_in_two_chunks_top16(kernel):
    """T = 512 at top_k = 16 is two launches of 256 tokens (4096 pairs each):
    every element of y against the oracle."""
    wl = Workload("prefill-k16", T=512, H=1024, I=512, E=64, k=16, routing="uniform", seed=21)
    x, ids, w = make_x(wl), make_topk_ids(wl), make_topk_w(wl)
    W = small_weights(wl)
    plan, ws, y, st = run_case(wl, x, ids, w, W, kernel=kernel)
    assert st == 0, binding.STATUS_NAMES.get(st)
    assert plan.stats()["prefill_launches"] == 2
    y_ref, _ = oracle.moe_forward(x, ids, w, {kk: v.cpu() for kk, v in W.items()})
    err = rel_err(y.cpu().numpy(), y_ref)
    print(f"prefill in two chunks at top_k=16: rel err {err:.3e}")
    assert err <= TOL


@pytest.mark.parametrize("name", ["decode", "spec_verify"])
def test_tensor_kernel_bitwise_reproducible(name, cache):
    wl, x, ids, w, W = workload_inputs(name, cache)
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=wl.T, strict=True, kernel=binding.MOE_KERNEL_TENSOR)
    ws = plan.new_workspace()
    xd, idd, wd = x.to(DEV), ids.to(DEV), w.to(DEV)
    y1 = plan.step(xd, idd, wd, ws).clone()
    y2 = plan.step(xd, idd, wd, ws).clone()
    assert plan.check(ws) == 0
    assert torch.equal(y1, y2)


# T = 17, 20: gate/up MMA N = 80 (per-token x rows); T = 33: per-pair x rows in
# one launch; E = 2: 24 pairs per expert, several groups of one expert;
# I = 4096: the largest I, 32 h slices per pair; H = 8192: two rounds of x loads
@pytest.mark.parametrize("T,H,I,E,k", [(1, 512, 256, 6, 3), (5, 512, 512, 6, 3), (12, 768, 768, 9, 4),
                                       (24, 512, 256, 16, 8), (17, 512, 512, 8, 4), (20, 768, 256, 12, 6),
                                       (33, 512, 256, 16, 8), (24, 512, 256, 2, 2), (12, 256, 4096, 4, 2),
                                       (4, 8192, 256, 4, 4)])
def test_tensor_kernel_small_shapes(T, H, I, E, k):
    wl = Workload("tc-small", T=T, H=H, I=I, E=E, k=k, routing="uniform", seed=11)
    ids = make_topk_ids(wl)
    x, w = make_x(wl), make_topk_w(wl)
    W = small_weights(wl)
    plan, ws, y, st = run_case(wl, x, ids, w, W, strict=False, kernel=binding.MOE_KERNEL_TENSOR)
    assert st == 0, binding.STATUS_NAMES.get(st)
    y_ref, _ = oracle.moe_forward(x, ids, w, {kk: v.cpu() for kk, v in W.items()})
    assert rel_err(y.cpu().numpy(), y_ref) <= TOL


def test_tensor_kernel_refuses_shapes_it_cannot_take():
    wl = Workload("tc-refuse", T=2, H=256, I=128, E=4, k=2, routing="uniform", seed=12)
    W = small_weights(wl)
    with pytest.raises(MoeError) as ei:
        MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=2, kernel=binding.MOE_KERNEL_TENSOR)
    assert ei.value.status == binding.MOE_ERR_UNSUPPORTED_SHAPE


def test_bitwise_reproducible(cache):
    wl, x, ids, w, W = workload_inputs("spec_verify", cache)
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=wl.T, strict=True)
    ws = plan.new_workspace()
    xd, idd, wd = x.to(DEV), ids.to(DEV), w.to(DEV)
    y1 = plan.step(xd, idd, wd, ws).clone()
    y2 = plan.step(xd, idd, wd, ws).clone()
    assert plan.check(ws) == 0
    assert torch.equal(y1, y2)


def test_token_permutation_permutes_output(cache):
    wl, x, ids, w, W = workload_inputs("spec_verify", cache)
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=wl.T, strict=True)
    ws = plan.new_workspace()
    p = torch.from_numpy(np.random.default_rng(3).permutation(wl.T))
    y = plan.step(x.to(DEV), ids.to(DEV), w.to(DEV), ws)
    yp = plan.step(x[p].contiguous().to(DEV), ids[p].contiguous().to(DEV), w[p].contiguous().to(DEV), ws)
    assert plan.check(ws) == 0
    assert torch.equal(yp, y[p.to(DEV)])


def test_zero_routing_weights_give_zero(cache):
    wl, x, ids, w, W = workload_inputs("decode", cache)
    _, _, y, st = run_case(wl, x, ids, torch.zeros_like(w), W)
    assert st == 0 and bool((y == 0).all())


@pytest.mark.parametrize("kernel,counter", [(binding.MOE_KERNEL_AUTO, "gemv_launches"),
                                            (binding.MOE_KERNEL_REGISTER, "decode_launches")])
def test_null_step_runs(cache, kernel, counter):
    """The measurement variant on the one-token row kernel (the automatic
    choice at T = 1) and on the register kernel."""
    wl, x, ids, w, W = workload_inputs("decode", cache)
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=wl.T, strict=True, kernel=kernel)
    ws = plan.new_workspace()
    plan.step(x.to(DEV), ids.to(DEV), w.to(DEV), ws, null=True)
    s = plan.stats()
    assert plan.check(ws) == 0 and s["null_launches"] == 1
    assert s["gemv_launches"] == (1 if counter == "gemv_launches" else 0)
    # the workspace counters are clean afterwards: a real step still matches
    y = plan.step(x.to(DEV), ids.to(DEV), w.to(DEV), ws)
    assert plan.stats()[counter] >= 1
    y_ref, _ = oracle.moe_forward(x, ids, w, weights_cpu(W, touched_experts(ids, wl.E)))
    assert rel_err(y.cpu().numpy(), y_ref) <= TOL


# ------------------------------------------------------------------ edge cases on small shapes
def small_weights(wl):
    return make_expert_weights(wl, device=DEV, experts=None)


def check_small(wl, ids, *, w=None, strict=False, T_max=None, expect_status=0, tokens=None):
    x = make_x(wl)
    w = make_topk_w(wl) if w is None else w
    W = small_weights(wl)
    plan, ws, y, st = run_case(wl, x, ids, w, W, strict=strict, T_max=T_max)
    assert st == expect_status, binding.STATUS_NAMES.get(st)
    Wc = {k: v.cpu() for k, v in W.items()}
    y_ref, _ = oracle.moe_forward(x, ids, w, Wc, tokens=tokens)
    yy = y.cpu().numpy() if tokens is None else y.cpu().numpy()[tokens]
    err = rel_err(yy, y_ref)
    assert err <= TOL, err
    return y, y_ref


@pytest.mark.parametrize("H,I", [(384, 256), (256, 384), (1152, 640)])
def test_ragged_shapes(H, I):
    wl = Workload("ragged", T=5, H=H, I=I, E=5, k=3, routing="uniform", seed=2)
    check_small(wl, make_topk_ids(wl))


# the pairs of a launch are grouped by one warp (P <= 32), by the rank sort of
# 32 < P <= 256 (tensor-core kernel) or by the counting sort above; T = 40 is a
# prefill launch
@pytest.mark.parametrize("T,k", [(6, 4), (12, 4), (24, 8), (40, 8)])
def test_empty_duplicate_and_bad_slots(T, k):
    wl = Workload("slots", T=T, H=256, I=256, E=11, k=k, routing="uniform", seed=3)
    ids = make_topk_ids(wl).clone()
    ids[0, 1] = -1            # empty slot
    ids[1, 2] = ids[1, 0]     # duplicate expert within a token
    ids[2, :] = -1            # token with no valid slot -> y == 0
    ids[3, 3] = wl.E + 2      # out of range: skipped and flagged
    ids[T - 1, 0] = -5        # another empty slot, in the last token
    y, _ = check_small(wl, ids, expect_status=binding.MOE_ERR_BAD_EXPERT_ID)
    assert bool((y[2] == 0).all())


@pytest.mark.parametrize("T", [1, 8, 24])
def test_all_tokens_one_expert(T):
    wl = Workload("hot", T=T, H=256, I=256, E=4, k=2, routing="uniform", seed=4)
    ids = torch.zeros((T, 2), dtype=torch.int32)
    ids[:, 1] = 1 + torch.arange(T, dtype=torch.int32) % 3
    check_small(wl, ids)


def test_expert_with_more_than_32_pairs_via_prefill():
    wl = Workload("hot40", T=40, H=256, I=256, E=4, k=2, routing="uniform", seed=5)
    ids = torch.zeros((40, 2), dtype=torch.int32)
    ids[:, 1] = 3
    check_small(wl, ids)


def test_prefill_chunking_top16():
    # top_k = 16 -> 256 tokens per launch; T = 300 takes two launches
    wl = Workload("chunks", T=300, H=256, I=128, E=32, k=16, routing="uniform", seed=6)
    check_small(wl, make_topk_ids(wl), tokens=[0, 1, 255, 256, 257, 299])


def test_max_decode_tokens_top16():
    wl = Workload("k16", T=24, H=512, I=256, E=64, k=16, routing="uniform", seed=8)
    check_small(wl, make_topk_ids(wl), strict=True)


def test_strict_mode_refuses_off_path_and_t0_noop():
    wl = Workload("strict", T=25, H=256, I=128, E=8, k=2, routing="uniform", seed=9)
    x, ids, w = make_x(wl), make_topk_ids(wl), make_topk_w(wl)
    W = small_weights(wl)
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=32, strict=True)
    ws = plan.new_workspace()
    y = torch.empty((wl.T, wl.H), dtype=torch.float32, device=DEV)
    with pytest.raises(MoeError) as ei:
        binding.moe_decode(plan.handle, x.to(DEV), ids.to(DEV), w.to(DEV), y, ws)
    assert ei.value.status == binding.MOE_ERR_NOT_FAST_PATH
    assert plan.stats()["rejected_calls"] == 1 and plan.stats()["decode_launches"] == 0
    # T == 0 is a no-op
    e0 = torch.empty((0, wl.H), dtype=torch.bfloat16, device=DEV)
    binding.moe_decode(plan.handle, e0, torch.empty((0, 2), dtype=torch.int32, device=DEV),
                       torch.empty((0, 2), dtype=torch.float32, device=DEV),
                       torch.empty((0, wl.H), dtype=torch.float32, device=DEV), ws)
    assert plan.stats()["decode_launches"] == 0
    # non-strict plans forward T > 24 to the prefill path
    plan2 = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=32, strict=False)
    binding.moe_decode(plan2.handle, x.to(DEV), ids.to(DEV), w.to(DEV), y, ws)
    assert plan2.check(ws) == 0 and plan2.stats()["prefill_launches"] == 1


def test_invalid_arguments_rejected_on_host():
    wl = Workload("args", T=2, H=256, I=128, E=8, k=2, routing="uniform", seed=10)
    W = small_weights(wl)
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=4)
    ws = plan.new_workspace()
    xb = torch.zeros(wl.T * wl.H + 8, dtype=torch.bfloat16, device=DEV)
    x_mis = xb[1:1 + wl.T * wl.H].view(wl.T, wl.H)       # 2-byte offset: misaligned
    ids = make_topk_ids(wl).to(DEV)
    w = make_topk_w(wl).to(DEV)
    y = torch.empty((wl.T, wl.H), dtype=torch.float32, device=DEV)
    with pytest.raises(MoeError) as ei:
        binding.moe_decode(plan.handle, x_mis, ids, w, y, ws)
    assert ei.value.status == binding.MOE_ERR_MISALIGNED
    with pytest.raises(MoeError) as ei:
        binding.moe_decode(plan.handle, torch.zeros((5, wl.H), dtype=torch.bfloat16, device=DEV),
                           torch.zeros((5, 2), dtype=torch.int32, device=DEV),
                           torch.zeros((5, 2), dtype=torch.float32, device=DEV),
                           torch.empty((5, wl.H), dtype=torch.float32, device=DEV), ws)
    assert ei.value.status == binding.MOE_ERR_INVALID_ARG     # T > T_max
    with pytest.raises(MoeError) as ei:
        MoePlan(W, 200, wl.I, wl.E, wl.k, T_max=4)             # H not a multiple of 128
    assert ei.value.status == binding.MOE_ERR_UNSUPPORTED_SHAPE
    # tensors that disagree about T or top_k are refused before the call
    x_ok = torch.zeros((wl.T, wl.H), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(MoeError) as ei:
        plan.step(x_ok, ids[:, :1].contiguous(), w[:, :1].contiguous(), ws)   # ids not [T, top_k]
    assert ei.value.status == binding.MOE_ERR_INVALID_ARG
    with pytest.raises(MoeError) as ei:
        binding.moe_decode(plan.handle, x_ok, ids[:1].contiguous(), w[:1].contiguous(), y, ws)   # 1 row of ids
    assert ei.value.status == binding.MOE_ERR_INVALID_ARG
    # moe_group with T * top_k beyond int range: refused before any launch
    i32 = dict(dtype=torch.int32, device=DEV)
    lib = binding.load_library()
    assert lib.moe_group(plan.handle, binding._ptr(ids), 1 << 30, binding._ptr(ws),
                         binding._ptr(torch.zeros(wl.E, **i32)), binding._ptr(torch.zeros(wl.E + 1, **i32)),
                         binding._ptr(torch.zeros(wl.T * wl.k, **i32)), None) == binding.MOE_ERR_INVALID_ARG
    assert plan.check(ws) == 0


# ------------------------------------------------------------------ grouping kernel, bit-exact
@pytest.mark.parametrize("T,k,E,seed", [(1, 8, 256, 0), (16, 8, 256, 1), (24, 8, 256, 2), (512, 8, 256, 3),
                                        (7, 4, 5, 4), (256, 16, 1024, 5)])
def test_grouping_bit_exact(T, k, E, seed):
    wl = Workload("g", T=1, H=128, I=128, E=E, k=k, routing="uniform")
    W = make_expert_weights(wl.replace(E=1), device=DEV)   # any valid plan weights
    plan = MoePlan(W, 128, 128, E, k, T_max=max(T, 1))
    ws = plan.new_workspace()
    rng = np.random.default_rng(seed)
    ids = torch.from_numpy(rng.integers(-1, E + 1, size=(T, k)).astype(np.int32))
    counts, offsets, perm = plan.group(ids.to(DEV), ws)
    rc, ro, rp, bad = oracle.group(ids, E)
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(perm.cpu().numpy(), rp)
    st = plan.check(ws)
    assert st == (binding.MOE_ERR_BAD_EXPERT_ID if bad else 0)


# ------------------------------------------------------------------ input recipe is device independent
def test_quantizer_identical_on_cpu_and_gpu():
    g = torch.Generator().manual_seed(11)
    w = torch.randn((512, 1024), generator=g) * 0.02
    a = quantize_nvfp4(w)
    b = quantize_nvfp4(w.to(DEV))
    assert torch.equal(a[0], b[0].cpu()) and torch.equal(a[1], b[1].cpu()) and float(a[2]) == float(b[2])


# ------------------------------------------------------------------ failure path: bounded waits
def test_poisoned_workspace_times_out_and_recovers():
    """A phase-A counter nothing will complete makes the bounded wait expire:
    the launch returns, moe_check reports MOE_ERR_TIMEOUT, and after
    moe_workspace_init the same plan computes correctly again."""
    os.environ["MOE_WAIT_TIMEOUT_MS"] = "200"
    try:
        wl = Workload("poison", T=2, H=256, I=128, E=8, k=2, routing="uniform", seed=12)
        x, ids, w = make_x(wl), make_topk_ids(wl), make_topk_w(wl)
        W = small_weights(wl)
        plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=wl.T)
    finally:
        del os.environ["MOE_WAIT_TIMEOUT_MS"]
    ws = plan.new_workspace()
    binding.moe_debug_poison_workspace(plan.handle, ws)
    plan.step(x.to(DEV), ids.to(DEV), w.to(DEV), ws)
    assert plan.check(ws) == binding.MOE_ERR_TIMEOUT
    binding.moe_workspace_init(plan.handle, ws)
    y = plan.step(x.to(DEV), ids.to(DEV), w.to(DEV), ws)
    assert plan.check(ws) == 0
    y_ref, _ = oracle.moe_forward(x, ids, w, {k: v.cpu() for k, v in W.items()})
    assert rel_err(y.cpu().numpy(), y_ref) <= TOL


def test_poisoned_workspace_times_out_and_recovers_tensor_kernel():
    """The same on the tensor-core kernel: with the gate/up counters poisoned no
    group's h is ever published, so the down tickets' waits expire; the launch
    returns (MMAs drained, tensor memory freed), moe_check reports the timeout, and
    after moe_workspace_init the plan computes correctly again."""
    os.environ["MOE_WAIT_TIMEOUT_MS"] = "200"
    try:
        wl = Workload("poison-tc", T=12, H=512, I=256, E=8, k=4, routing="uniform", seed=13)
        x, ids, w = make_x(wl), make_topk_ids(wl), make_topk_w(wl)
        W = small_weights(wl)
        plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=wl.T)
    finally:
        del os.environ["MOE_WAIT_TIMEOUT_MS"]
    ws = plan.new_workspace()
    binding.moe_debug_poison_workspace(plan.handle, ws)
    plan.step(x.to(DEV), ids.to(DEV), w.to(DEV), ws)
    assert plan.check(ws) == binding.MOE_ERR_TIMEOUT
    assert plan.stats()["tensor_launches"] == 1
    binding.moe_workspace_init(plan.handle, ws)
    y = plan.step(x.to(DEV), ids.to(DEV), w.to(DEV), ws)
    assert plan.check(ws) == 0
    y_ref, _ = oracle.moe_forward(x, ids, w, {k: v.cpu() for k, v in W.items()})
    assert rel_err(y.cpu().numpy(), y_ref) <= TOL


def test_poisoned_workspace_times_out_and_recovers_small_kernel():
    """The same on the small-launch tensor-core kernel: with the experts'
    gate/up counters poisoned no h is ever built, so the waits of the down
    groups expire; the launch returns (copies drained, MMAs complete, tensor
    memory freed), moe_check reports the timeout, and after moe_workspace_init
    the plan computes correctly again."""
    os.environ["MOE_WAIT_TIMEOUT_MS"] = "200"
    try:
        wl = Workload("poison-small", T=2, H=512, I=256, E=8, k=4, routing="uniform", seed=14)
        x, ids, w = make_x(wl), make_topk_ids(wl), make_topk_w(wl)
        W = small_weights(wl)
        plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=wl.T)
    finally:
        del os.environ["MOE_WAIT_TIMEOUT_MS"]
    ws = plan.new_workspace()
    binding.moe_debug_poison_workspace(plan.handle, ws)
    plan.step(x.to(DEV), ids.to(DEV), w.to(DEV), ws)
    assert plan.check(ws) == binding.MOE_ERR_TIMEOUT
    assert plan.stats()["small_launches"] == 1
    binding.moe_workspace_init(plan.handle, ws)
    y = plan.step(x.to(DEV), ids.to(DEV), w.to(DEV), ws)
    assert plan.check(ws) == 0
    y_ref, _ = oracle.moe_forward(x, ids, w, {k: v.cpu() for k, v in W.items()})
    assert rel_err(y.cpu().numpy(), y_ref) <= TOL


# ------------------------------------------------------------------ programmatic dependent launch
def test_pdl_back_to_back_matches(cache):
    """Steps launched with programmatic dependent launch, back to back on one
    stream over a shared workspace, give the same bits as plain launches."""
    wl, x, ids, w, W = workload_inputs("spec_verify", cache)
    ref_plan, ref_ws, y_ref, st = run_case(wl, x, ids, w, W)
    assert st == 0
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=wl.T, strict=True, pdl=True)
    ws = plan.new_workspace()
    xd, idsd, wd = x.to(DEV), ids.to(DEV), w.to(DEV)
    ys = [torch.empty((wl.T, wl.H), dtype=torch.float32, device=DEV) for _ in range(4)]
    for y in ys:
        plan.step(xd, idsd, wd, ws, y=y)
    assert plan.check(ws) == 0
    for y in ys:
        assert torch.equal(y, y_ref)
