"""GB300-native row-wise RMSNorm hot path.

Two operations, hand-written CUDA for sm_103a behind the C ABI of
include/rmsnorm.h (librmsnorm_gb300.so), with these thin Python bindings:

  rmsnorm_fwd  -- fused residual-add RMSNorm forward with two outputs
                  (out, new_residual), fp32 accumulation, weight_bias scalar.
  rmsnorm_fwd_bind, rmsnorm_vjp_bind -- the same calls with their tensors
                  checked once, for loops over fixed buffers (decode).
  rmsnorm_vjp  -- RMSNorm VJP: gx and an fp32 gw reduced across rows inside
                  the kernels (deterministic, no [rows, D] temporary).
  rmsnorm_fused_vjp -- VJP of the two-output fused op (adds the gradient that
                  reaches new_residual in the same pass).
  rmsnorm_fwd_ex, rmsnorm_vjp_ex -- the same on rows a stride apart, with the
                  forward's per-row scale (rstd) written and reused.
  fp16, bf16 and fp32 tensors.
  fused_add_rmsnorm, rms_norm -- torch.autograd wrappers.
  rmsnorm_gated_silu -- the decode loop's gated activation silu(x[:d]) * x[d:].
  rmsnorm_rope_kv_append -- rotary embedding of q and k with the KV-cache append.

PyTorch supplies device memory and streams only.
"""
from .api import (  # noqa: F401
    BoundCall,
    rmsnorm_debug_claim_counters,
    rmsnorm_debug_fail_allocs,
    rmsnorm_debug_inject,
    rmsnorm_describe_dispatch,
    rmsnorm_device_status,
    rmsnorm_fused_vjp,
    rmsnorm_fwd,
    rmsnorm_fwd_bind,
    rmsnorm_fwd_ex,
    rmsnorm_gated_silu,
    rmsnorm_rope_kv_append,
    rmsnorm_status_string,
    rmsnorm_vjp,
    rmsnorm_vjp_bind,
    rmsnorm_vjp_ex,
    rmsnorm_vjp_noalloc,
    rmsnorm_vjp_workspace_size,
    rmsnorm_vjp_ws,
)
from ._native import DEVSTATUS_BAD_INDEX, DEVSTATUS_WAIT_TIMEOUT, MAX_D, RmsnormError  # noqa: F401
from .autograd import fused_add_rmsnorm, rms_norm  # noqa: F401

__all__ = [
    "rmsnorm_fwd",
    "rmsnorm_vjp",
    "rmsnorm_fwd_bind",
    "rmsnorm_vjp_bind",
    "BoundCall",
    "rmsnorm_fused_vjp",
    "rmsnorm_fwd_ex",
    "rmsnorm_vjp_ex",
    "rmsnorm_gated_silu",
    "rmsnorm_rope_kv_append",
    "fused_add_rmsnorm",
    "rms_norm",
    "rmsnorm_vjp_ws",
    "rmsnorm_vjp_noalloc",
    "rmsnorm_vjp_workspace_size",
    "rmsnorm_device_status",
    "rmsnorm_debug_inject",
    "rmsnorm_debug_fail_allocs",
    "rmsnorm_debug_claim_counters",
    "rmsnorm_describe_dispatch",
    "rmsnorm_status_string",
    "RmsnormError",
]
