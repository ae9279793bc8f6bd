"""GB300 (sm_103a) routed-experts MoE step over NVFP4 expert weights.

The computation runs in libmoe_nvfp4.so (include/moe_nvfp4.h); `binding`
marshals torch CUDA tensors into it; `inputs` draws the seeded synthetic
workloads.  Build the library with `quantized_moe_routed_gb300.build.build()`.
"""
from .binding import (ABI_SYMBOLS, HostIO, MoeError, MoePlan, expert_range, load_library, moe_abi_version, moe_check,  # noqa: F401
                      moe_debug_poison_workspace, moe_decode, moe_step_host, moe_decode_static, moe_group,
                      moe_io_bytes, moe_last_error, moe_null_step, moe_plan_create, moe_plan_destroy, moe_prefill,
                      moe_route, moe_stats, moe_status_string, moe_workspace_bytes, moe_workspace_init)
