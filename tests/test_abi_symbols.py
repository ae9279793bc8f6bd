"""The C-ABI library loads and exports every function include/moe_nvfp4.h
declares, and the binding prototypes exactly those (no GPU needed)."""
import ctypes
import os
import re

from conftest import ROOT


def _declared():
    src = open(os.path.join(ROOT, "include", "moe_nvfp4.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src))


def test_library_exports_every_declared_symbol():
    from quantized_moe_routed_gb300 import build as libbuild
    from quantized_moe_routed_gb300 import binding
    path = libbuild.build()
    decl = _declared()
    assert decl == set(binding.ABI_SYMBOLS), decl ^ set(binding.ABI_SYMBOLS)
    lib = ctypes.CDLL(path)
    for name in decl:
        assert hasattr(lib, name), name
    lib.moe_abi_version.restype = ctypes.c_int
    assert lib.moe_abi_version() == 8
    lib.moe_status_string.restype = ctypes.c_char_p
    assert lib.moe_status_string(6) == b"MOE_ERR_TIMEOUT"


def test_plan_desc_and_stats_match_the_header():
    # the ctypes mirrors of moe_plan_desc / moe_stats_t list the header's fields in order
    from quantized_moe_routed_gb300 import binding
    src = open(os.path.join(ROOT, "include", "moe_nvfp4.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    for struct, py in (("moe_plan_desc", binding.moe_plan_desc), ("moe_stats_t", binding.moe_stats_t)):
        body = re.search(r"typedef struct \{([^{}]*)\}\s*" + struct + ";", src).group(1)
        names = re.findall(r"\*?\s*(\w+)\s*[,;]", body)
        assert names == [f for f, _ in py._fields_], (struct, names)
    assert (binding.MOE_KERNEL_AUTO, binding.MOE_KERNEL_REGISTER, binding.MOE_KERNEL_TENSOR) == (0, 1, 2)


def test_binding_loads_and_rejects_without_plan():
    import quantized_moe_routed_gb300 as q
    lib = q.load_library()
    # host-side validation needs no GPU: a null plan is rejected with a message
    assert lib.moe_check(None, None, None) == q.binding.MOE_ERR_INVALID_ARG
    assert "null" in q.moe_last_error()
    assert q.moe_workspace_bytes(None, 1) == 0
    assert q.moe_io_bytes(None, 1) == (0, 0, 0)
    assert lib.moe_step_host(None, None, None, None, None, 1, None, None) == q.binding.MOE_ERR_INVALID_ARG
    assert lib.moe_route(None, None, 1, None, None, None) == q.binding.MOE_ERR_INVALID_ARG


def test_step_shapes_must_agree():
    # the binding refuses tensors that disagree about T, top_k or H before any call
    import pytest
    import torch
    from quantized_moe_routed_gb300 import MoeError, binding
    T, H, k = 3, 256, 4
    x, ids, w, y = (torch.zeros((T, H)), torch.zeros((T, k)), torch.zeros((T, k)), torch.zeros((T, H)))
    binding._need_step_shapes(x, ids, w, y)
    binding._need_step_shapes(x, ids, w, torch.zeros((T + 2, H)))          # a taller y is fine
    binding._need_step_shapes(torch.zeros((0, H)), torch.zeros((0, k)), torch.zeros((0, k)), torch.zeros((0, H)))
    bad = [(x, ids[:1], w[:1], y), (x, ids, w[:, :2], y), (x, ids, w, y[:1]), (x, ids, w, torch.zeros((T, H + 1))),
           (x.reshape(-1), ids, w, y), (x, ids.reshape(-1), w.reshape(-1), y)]
    for args in bad:
        with pytest.raises(MoeError) as ei:
            binding._need_step_shapes(*args)
        assert ei.value.status == binding.MOE_ERR_INVALID_ARG
