"""GB300-native row-wise RMSNorm hot path.

Two operations, hand-written CUDA for sm_103a behind the C ABI of
include/rmsnorm.h (librmsnorm_gb300.so), with these thin Python bindings:

  rmsnorm_fwd  -- fused residual-add RMSNorm forward with two outputs
                  (out, new_residual), fp32 accumulation, weight_bias scalar.
  rmsnorm_vjp  -- RMSNorm VJP: gx and an fp32 gw reduced across rows inside
                  the kernels (deterministic, no [rows, D] temporary).

PyTorch supplies device memory and streams only.
"""
from .api import (  # noqa: F401
    rmsnorm_debug_inject,
    rmsnorm_describe_dispatch,
    rmsnorm_device_status,
    rmsnorm_fwd,
    rmsnorm_status_string,
    rmsnorm_vjp,
    rmsnorm_vjp_workspace_size,
    rmsnorm_vjp_ws,
)
from ._native import DEVSTATUS_WAIT_TIMEOUT, MAX_D, RmsnormError  # noqa: F401

__all__ = [
    "rmsnorm_fwd",
    "rmsnorm_vjp",
    "rmsnorm_vjp_ws",
    "rmsnorm_vjp_workspace_size",
    "rmsnorm_device_status",
    "rmsnorm_debug_inject",
    "rmsnorm_describe_dispatch",
    "rmsnorm_status_string",
    "RmsnormError",
]
