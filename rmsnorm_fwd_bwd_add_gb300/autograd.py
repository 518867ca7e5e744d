"""torch.autograd wrappers over the C ABI.

fused_add_rmsnorm(x, residual, w, eps, weight_bias) -> (out, new_residual)
    forward: rmsnorm_fwd_ex, which also saves each row's scale (rstd);
    backward: rmsnorm_vjp_ex on the saved new_residual with that rstd, giving
    one gradient for x and residual (they enter as a sum) and gw.
rms_norm(x, w, eps, weight_bias) -> out
    forward: rmsnorm_fwd_ex without a residual; backward: rmsnorm_vjp_ex.
Inputs whose rows sit a stride apart (slices of wider buffers) are used in
place; fp16, bf16 and fp32.

The kernels accumulate gw in fp32; it is returned in w's dtype, as autograd
expects a gradient of a parameter's own dtype.  Gradients that do not reach
an output arrive as None and are not materialised.

Source: "Fused residual-add RMSNorm and fused RoPE + KV-append decode
kernels", Background (two-output FusedAddRMSNorm); "RMSNormVJP backward
writes a full {n_rows, D} gw_temp intermediate", POC (the gradients of
rms_norm through autograd).
"""
from __future__ import annotations

import torch

from .api import rmsnorm_fwd_ex, rmsnorm_vjp_ex, rows_layout_ok


def _rows(t):
    """t itself when the kernels take its layout (rows a stride apart), else a
    dense copy (e.g. an expanded gradient of a sum)."""
    return t if rows_layout_ok(t) else t.contiguous()


class FusedAddRMSNormFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, residual, w, eps: float, weight_bias: float):
        ctx.set_materialize_grads(False)
        out, new_res, rstd = rmsnorm_fwd_ex(_rows(x), w.contiguous(), eps, weight_bias,
                                            _rows(residual), rstd=True)
        ctx.save_for_backward(new_res, w, rstd)
        ctx.eps = eps
        ctx.weight_bias = weight_bias
        return out, new_res

    @staticmethod
    def backward(ctx, g_out, g_res):
        new_res, w, rstd = ctx.saved_tensors
        if g_out is None:
            g_h = None if g_res is None else g_res.contiguous()
            gw = torch.zeros_like(w) if ctx.needs_input_grad[2] else None
        else:
            g_h, gw32 = rmsnorm_vjp_ex(new_res, w.contiguous(), _rows(g_out), ctx.eps,
                                       ctx.weight_bias, None if g_res is None else _rows(g_res),
                                       rstd=rstd)
            gw = gw32.to(w.dtype) if ctx.needs_input_grad[2] else None
        gx = g_h if ctx.needs_input_grad[0] else None
        gr = g_h if ctx.needs_input_grad[1] else None
        return gx, gr, gw, None, None


class RMSNormFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, w, eps: float, weight_bias: float):
        x = _rows(x)
        out, _, rstd = rmsnorm_fwd_ex(x, w.contiguous(), eps, weight_bias, rstd=True)
        ctx.save_for_backward(x, w, rstd)
        ctx.eps = eps
        ctx.weight_bias = weight_bias
        return out

    @staticmethod
    def backward(ctx, g_out):
        x, w, rstd = ctx.saved_tensors
        gx, gw32 = rmsnorm_vjp_ex(x, w.contiguous(), _rows(g_out), ctx.eps, ctx.weight_bias,
                                  rstd=rstd)
        return (gx if ctx.needs_input_grad[0] else None,
                gw32.to(w.dtype) if ctx.needs_input_grad[1] else None, None, None)


def fused_add_rmsnorm(x, residual, w, eps: float, weight_bias: float = 0.0):
    """(out, new_residual) with h = x + residual and
    out = h * rsqrt(mean(h^2) + eps) * (weight_bias + w); differentiable."""
    return FusedAddRMSNormFunction.apply(x, residual, w, eps, weight_bias)


def rms_norm(x, w, eps: float, weight_bias: float = 0.0):
    """x * rsqrt(mean(x^2) + eps) * (weight_bias + w); differentiable."""
    return RMSNormFunction.apply(x, w, eps, weight_bias)
