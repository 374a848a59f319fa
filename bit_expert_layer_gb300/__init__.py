"""GB300 (sm_103a) library for the mixture-of-experts layer of Qwen3.6-35B-A3B over
MLX affine 4-bit (group-64) expert weights.

The compute lives in ``libmoe_layer.so`` (hand-written CUDA, C ABI in
``include/moe_layer.h``); this package is a ctypes binding (``_abi``, same names as
the C entry points) plus torch-facing wrappers (``layer``).  Build with
``bit_expert_layer_gb300.build.build()``.
"""
from . import _abi
from ._abi import (MoEError, MoeConfig, MoeQMat, MoeWeights, moe_forward, moe_forward_launches,
                   moe_forward_residual, moe_layer_create, moe_layer_destroy, moe_layer_get_error, moe_route,
                   moe_stack_forward, moe_stack_forward_host, moe_status_string, moe_workspace_bytes)

__all__ = [
    "_abi", "MoEError", "MoeConfig", "MoeQMat", "MoeWeights", "moe_forward", "moe_forward_launches",
    "moe_forward_residual", "moe_layer_create", "moe_layer_destroy", "moe_layer_get_error", "moe_route",
    "moe_stack_forward", "moe_stack_forward_host", "moe_status_string", "moe_workspace_bytes",
]
