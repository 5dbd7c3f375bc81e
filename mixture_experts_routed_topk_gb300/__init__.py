"""Routed top-k mixture-of-experts expert layer (forward) for GB300 (sm_103a).

The compute path is the C-ABI library ``libmoe_gb300.so`` (hand-written CUDA kernels); the
functions re-exported here are its thin ctypes binding. Importing this package does not load the
library: the first call does, and it raises if the library has not been built.
"""

__all__ = [
    "moe_workspace_bytes",
    "moe_workspace_layout",
    "moe_routing_workspace_bytes",
    "moe_routing",
    "moe_fwd_dispatch",
    "moe_fwd_gemm1",
    "moe_fwd_gemm2",
    "moe_fwd_combine",
    "moe_routed_experts_fwd",
    "moe_routed_experts_fwd_rmsnorm",
    "moe_mega_workspace_bytes",
    "moe_mega_workspace_layout",
    "moe_routed_experts_fwd_mega",
    "moe_fwd_mega_stages",
    "moe_bwd_workspace_bytes",
    "moe_routed_experts_bwd",
    "moe_mxfp8_weight_bytes",
    "moe_mxfp8_prepare_weight",
    "moe_mxfp8_workspace_bytes",
    "moe_mxfp8_workspace_layout",
    "moe_routed_experts_fwd_mxfp8",
    "moe_fwd_mxfp8_stages",
    "moe_nvfp4_weight_bytes",
    "moe_nvfp4_prepare_weight",
    "moe_nvfp4_workspace_bytes",
    "moe_nvfp4_workspace_layout",
    "moe_routed_experts_fwd_nvfp4",
    "moe_fwd_nvfp4_stages",
    "MOE_WEIGHT_W13",
    "MOE_WEIGHT_W2",
    "moe_get_status",
    "moe_status_string",
    "MoeError",
    "alloc_workspace",
]


def __getattr__(name):
    if name in __all__:
        from . import binding

        return getattr(binding, name)
    raise AttributeError(name)
