"""The host-buffer entry (moe_step_host): one copy of the packed x / ids / w
block in (none for the one-token row kernel, which reads the pinned block in
place), then the step, which stores y straight into a pinned host y (or into
y_dev, with one copy out, when y is pageable).  Its result is bitwise the
result of the same step on device buffers, on every path it routes to
(register kernel, tensor-core kernel, prefill), and it refuses bad arguments
before it copies anything."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from quantized_moe_routed_gb300 import HostIO, MoeError, MoePlan, binding
from quantized_moe_routed_gb300.inputs import Workload, make_expert_weights, make_topk_ids, make_topk_w, make_x

pytestmark = pytest.mark.gpu
TOL = 2e-3
DEV = "cuda:0"


def rel_err(y, y_ref):
    y = np.asarray(y, dtype=np.float64)
    return float(np.abs(y - y_ref).max() / np.abs(y_ref).max())


def fill(io, x, ids, w):
    io.x.copy_(x)
    io.ids.copy_(ids)
    io.w.copy_(w)


# T = 1 x top-8: the small-launch tensor-core kernel at H = 512, the one-token
# row kernel at H = 2048 (and the register kernel on a register plan);
# T = 12 x top-4: the tensor-core ticket kernel; T = 40: the prefill path (a
# strict plan takes it through this entry)
@pytest.mark.parametrize("T,k,path", [(1, 8, "small"), (1, 8, "gemv"), (1, 8, "register"), (12, 4, "tensor"),
                                      (40, 4, "prefill")])
def test_step_host_is_bitwise_the_device_step(T, k, path):
    wl = Workload("hostio", T=T, H=2048 if path == "gemv" else 512, I=256, E=16, k=k, routing="uniform", seed=21)
    x, ids, w = make_x(wl), make_topk_ids(wl), make_topk_w(wl)
    W = make_expert_weights(wl, device=DEV, experts=None)
    kern = binding.MOE_KERNEL_REGISTER if path == "register" else binding.MOE_KERNEL_AUTO
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=T, strict=True, kernel=kern)
    ws = plan.new_workspace()
    y_dev_path = plan.step(x.to(DEV), ids.to(DEV), w.to(DEV), ws)
    assert plan.check(ws) == 0
    before = plan.stats()
    io = HostIO(plan, T)
    fill(io, x, ids, w)
    io.y_dev.fill_(float("nan"))
    io.dev.fill_(0xAB)
    y = plan.step_host(io, ws)
    torch.cuda.synchronize()
    assert plan.check(ws) == 0
    after = plan.stats()
    assert torch.equal(y, y_dev_path.cpu())
    # the pinned y is device-addressable: the kernels stored y there directly
    assert bool(torch.isnan(io.y_dev).all())
    # the row kernel reads the pinned input block in place; every other path copies it
    if path == "gemv":
        assert bool((io.dev == 0xAB).all())
    else:
        assert torch.equal(io.dev.cpu(), io.host)
    if path == "tensor":
        assert after["tensor_launches"] == before["tensor_launches"] + 1
    elif path == "small":
        assert after["small_launches"] == before["small_launches"] + 1
    elif path == "gemv":
        assert after["gemv_launches"] == before["gemv_launches"] + 1
    elif path == "register":
        assert after["tensor_launches"] == before["tensor_launches"]
        assert after["decode_launches"] == before["decode_launches"] + 1
    else:
        assert after["prefill_launches"] == before["prefill_launches"] + 1
    y_ref, _ = oracle.moe_forward(x, ids, w, {n: v.cpu() for n, v in W.items()})
    assert rel_err(y.numpy(), y_ref) <= TOL


def test_steps_queued_back_to_back_on_separate_blocks():
    """Four steps with different ids, each on its own block, queued without a
    synchronisation in between (one workspace, programmatic dependent launch):
    each y is the device-path result of its own inputs."""
    wl = Workload("hostio4", T=4, H=512, I=256, E=16, k=4, routing="uniform", seed=22)
    x, w = make_x(wl), make_topk_w(wl)
    W = make_expert_weights(wl, device=DEV, experts=None)
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=wl.T, strict=True, pdl=True)
    ws = plan.new_workspace()
    idss = [(make_topk_ids(wl) + s) % wl.E for s in range(4)]
    ios = []
    for ids in idss:
        io = HostIO(plan, wl.T)
        fill(io, x, ids, w)
        ios.append(io)
    for io in ios:
        plan.step_host(io, ws)
    torch.cuda.synchronize()
    assert plan.check(ws) == 0
    for io, ids in zip(ios, idss):
        y_ref = plan.step(x.to(DEV), ids.to(DEV), w.to(DEV), ws)
        assert torch.equal(io.y, y_ref.cpu())


def test_pageable_host_buffers_take_the_copies():
    """Pageable host buffers: the input block is staged by the runtime and y
    comes back by a copy from y_dev; the result is the same bits."""
    wl = Workload("hostio_p", T=2, H=512, I=256, E=8, k=4, routing="uniform", seed=25)
    x, ids, w = make_x(wl), make_topk_ids(wl), make_topk_w(wl)
    W = make_expert_weights(wl, device=DEV, experts=None)
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=wl.T, strict=True)
    ws = plan.new_workspace()
    y_ref = plan.step(x.to(DEV), ids.to(DEV), w.to(DEV), ws)
    n, oi, ow = binding.moe_io_bytes(plan.handle, wl.T)
    host = torch.zeros(n, dtype=torch.uint8)                # not pinned
    host[:x.numel() * 2].view(torch.bfloat16).copy_(x.reshape(-1))
    host[oi:oi + ids.numel() * 4].view(torch.int32).copy_(ids.reshape(-1))
    host[ow:ow + w.numel() * 4].view(torch.float32).copy_(w.reshape(-1))
    dev = torch.empty(n, dtype=torch.uint8, device=DEV)
    y_dev = torch.full((wl.T, wl.H), float("nan"), dtype=torch.float32, device=DEV)
    y_host = torch.zeros((wl.T, wl.H), dtype=torch.float32)  # not pinned
    binding.moe_step_host(plan.handle, host, dev, y_dev, y_host, wl.T, ws)
    torch.cuda.synchronize()
    assert plan.check(ws) == 0
    assert torch.equal(y_dev, y_ref) and torch.equal(y_host, y_ref.cpu())


def test_io_layout_and_shared_y():
    wl = Workload("hostio_l", T=3, H=512, I=256, E=8, k=8, routing="uniform", seed=23)
    W = make_expert_weights(wl, device=DEV, experts=None)
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=6)
    # x = 3 * 512 * 2 = 3072 bytes; ids and w 96 bytes each, each rounded up to 256
    assert binding.moe_io_bytes(plan.handle, 3) == (3584, 3072, 3328)
    assert binding.moe_io_bytes(plan.handle, 0)[0] == 0
    assert binding.moe_io_bytes(plan.handle, 7)[0] == 0
    a = HostIO(plan, 6)
    b = HostIO(plan, 3, y_from=a)
    assert b.y.data_ptr() == a.y.data_ptr() and b.y.shape == (3, 512)
    with pytest.raises(MoeError):
        HostIO(plan, 6, y_from=b)


def test_step_host_rejects_before_copying():
    wl = Workload("hostio_r", T=2, H=256, I=128, E=8, k=2, routing="uniform", seed=24)
    x, ids, w = make_x(wl), make_topk_ids(wl), make_topk_w(wl)
    W = make_expert_weights(wl, device=DEV, experts=None)
    plan = MoePlan(W, wl.H, wl.I, wl.E, wl.k, T_max=4)
    ws = plan.new_workspace()
    io = HostIO(plan, wl.T)
    fill(io, x, ids, w)
    io.dev.fill_(0xAB)
    yb = torch.empty(wl.T * wl.H + 4, dtype=torch.float32, device=DEV)
    y_mis = yb[1:1 + wl.T * wl.H].view(wl.T, wl.H)          # 4-byte offset: misaligned
    with pytest.raises(MoeError) as ei:
        binding.moe_step_host(plan.handle, io.host, io.dev, y_mis, io.y, wl.T, ws)
    assert ei.value.status == binding.MOE_ERR_MISALIGNED
    lib = binding.load_library()
    P = ctypes.c_void_p
    # through the C entry itself: T > T_max, a null host block, a null workspace
    assert lib.moe_step_host(plan.handle, P(io.host.data_ptr()), P(io.dev.data_ptr()), P(io.y_dev.data_ptr()),
                             P(io.y.data_ptr()), 5, P(ws.data_ptr()), None) == binding.MOE_ERR_INVALID_ARG
    assert lib.moe_step_host(plan.handle, None, P(io.dev.data_ptr()), P(io.y_dev.data_ptr()),
                             P(io.y.data_ptr()), wl.T, P(ws.data_ptr()), None) == binding.MOE_ERR_INVALID_ARG
    assert lib.moe_step_host(plan.handle, P(io.host.data_ptr()), P(io.dev.data_ptr()), P(io.y_dev.data_ptr()),
                             P(io.y.data_ptr()), wl.T, None, None) == binding.MOE_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool((io.dev == 0xAB).all())                     # nothing was copied
    assert plan.stats()["rejected_calls"] == 4
    # T == 0 is a no-op
    assert lib.moe_step_host(plan.handle, None, None, None, None, 0, None, None) == binding.MOE_OK
