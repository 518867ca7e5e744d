"""The two-output fused op's VJP (rmsnorm_fused_vjp) and the autograd wrappers
against the fp64 oracle.  Inputs follow the prefill recipe (configuration 4)
plus edge shapes that reach every tier."""
import numpy as np
import pytest
import torch

import oracle
import rmsnorm_fwd_bwd_add_gb300 as rn
from rmsnorm_fwd_bwd_add_gb300 import workloads as W
from parity import (assert_close, assert_close_conditioned, f64, gx_term_magnitude)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _library():
    from rmsnorm_fwd_bwd_add_gb300 import build
    build.build()
    yield
    assert rn.rmsnorm_device_status(clear=True) == 0


def _g_res(case, seed):
    gen = torch.Generator().manual_seed(seed)
    return torch.randn(case.rows, case.D, generator=gen).to(case.dtype)


def _rounded_h(case):
    _, h = oracle.fwd(f64(case.x), f64(case.w), case.eps, case.weight_bias, f64(case.residual))
    return torch.from_numpy(h).to(case.dtype)


@pytest.mark.parametrize("D", W.PREFILL_D)
def test_fused_vjp_prefill(D):
    case = W.config4(D, rows=4096)
    h = _rounded_h(case)
    g_res = _g_res(case, D)
    assert rn.rmsnorm_describe_dispatch("vjp", case.rows, D, case.dtype, True).startswith("staged")
    g_h, gw = rn.rmsnorm_fused_vjp(h.to(DEV), case.w.to(DEV), case.g.to(DEV), case.eps,
                                   case.weight_bias, g_res.to(DEV))
    want_gh, want_gw = oracle.fused_vjp(f64(h), f64(case.w), f64(case.g), case.eps,
                                        case.weight_bias, f64(g_res))
    assert_close("fused g_h", g_h, want_gh)
    assert_close("fused gw", gw, want_gw, torch.float32)


EDGE = [(1, 64), (3, 4096), (8, 8192), (9, 264), (300, 520), (1000, 1024), (157, 2048),
        (77, 33), (5, 1001), (11, 40000), (153, 16384), (263, 3072), (67, 12288), (99, 1536),
        (201, 2560), (109, 3584), (87, 5120), (45, 7168)]


@pytest.mark.parametrize("rows,D", EDGE, ids=["r%d_d%d" % e for e in EDGE])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_fused_vjp_edges(rows, D, dtype):
    case = W.random_case(rows, D, dtype, seed=rows * 31 + D, weight_bias=1.0, eps=1e-5)
    h = _rounded_h(case)
    g_res = _g_res(case, rows + D)
    g_h, gw = rn.rmsnorm_fused_vjp(h.to(DEV), case.w.to(DEV), case.g.to(DEV), case.eps,
                                   case.weight_bias, g_res.to(DEV))
    want_gh, want_gw = oracle.fused_vjp(f64(h), f64(case.w), f64(case.g), case.eps,
                                        case.weight_bias, f64(g_res))
    terms = gx_term_magnitude(h, case.w, case.g, case.eps, case.weight_bias) + np.abs(f64(g_res))
    assert_close_conditioned("fused g_h", g_h, want_gh, terms)
    assert_close("fused gw", gw, want_gw, torch.float32)


def test_fused_vjp_without_residual_gradient_is_the_vjp():
    case = W.config4(4096, rows=1024)
    h = _rounded_h(case).to(DEV)
    w, g = case.w.to(DEV), case.g.to(DEV)
    a = rn.rmsnorm_fused_vjp(h, w, g, case.eps, 0.0, None)
    b = rn.rmsnorm_vjp(h, w, g, case.eps, 0.0)
    assert torch.equal(a[0], b[0])
    assert torch.equal(a[1].view(torch.int32), b[1].view(torch.int32))


def test_fused_vjp_in_place_over_g_out():
    case = W.config4(8192, rows=512)
    h = _rounded_h(case)
    g_res = _g_res(case, 5)
    want_gh, want_gw = oracle.fused_vjp(f64(h), f64(case.w), f64(case.g), case.eps,
                                        case.weight_bias, f64(g_res))
    g = case.g.to(DEV)
    g_h, gw = rn.rmsnorm_fused_vjp(h.to(DEV), case.w.to(DEV), g, case.eps, case.weight_bias,
                                   g_res.to(DEV), g_h=g)
    assert g_h.data_ptr() == g.data_ptr()
    assert_close("in-place g_h", g, want_gh)
    assert_close("in-place gw", gw, want_gw, torch.float32)


@pytest.mark.parametrize("rows,D,wb", [(2048, 4096, 0.0), (6, 8192, 1.0), (300, 512, 0.0)])
def test_autograd_fused_add_rmsnorm(rows, D, wb):
    case = W.random_case(rows, D, torch.bfloat16, seed=rows, weight_bias=wb)
    x = case.x.to(DEV).requires_grad_()
    res = case.residual.to(DEV).requires_grad_()
    w = case.w.to(DEV).requires_grad_()
    out, new_res = rn.fused_add_rmsnorm(x, res, w, case.eps, wb)
    g_out = case.g.to(DEV)
    g_res = _g_res(case, 99).to(DEV)
    loss = (out.float() * g_out.float()).sum() + (new_res.float() * g_res.float()).sum()
    gx, gr, gw = torch.autograd.grad(loss, (x, res, w))
    # autograd routes g_out / g_res back as the loss's gradients of out / new_res
    h = _rounded_h(case)
    want_gh, want_gw = oracle.fused_vjp(f64(h), f64(case.w), f64(case.g), case.eps, wb,
                                        f64(g_res.cpu()))
    assert_close("autograd dx", gx, want_gh)
    assert torch.equal(gx, gr)
    assert gw.dtype == w.dtype
    assert_close("autograd dw", gw, want_gw)


def test_autograd_only_out_used():
    case = W.random_case(512, 1024, torch.bfloat16, seed=7)
    x = case.x.to(DEV).requires_grad_()
    res = case.residual.to(DEV).requires_grad_()
    w = case.w.to(DEV).requires_grad_()
    out, _ = rn.fused_add_rmsnorm(x, res, w, case.eps)
    (gx,) = torch.autograd.grad((out.float() * case.g.to(DEV).float()).sum(), (x,))
    h = _rounded_h(case)
    want_gh, _ = oracle.vjp(f64(h), f64(case.w), f64(case.g), case.eps, case.weight_bias)
    assert_close("autograd dx (out only)", gx, want_gh)


def test_autograd_rms_norm():
    case = W.config1()
    x = case.x.to(DEV).requires_grad_()
    w = case.w.to(DEV).requires_grad_()
    out = rn.rms_norm(x, w, case.eps)
    want_out, _ = oracle.fwd(f64(case.x), f64(case.w), case.eps)
    assert_close("rms_norm out", out, want_out)
    gx, gw = torch.autograd.grad((out.float() * case.g.to(DEV).float()).sum(), (x, w))
    want_gx, want_gw = oracle.vjp(f64(case.x), f64(case.w), f64(case.g), case.eps)
    assert_close("rms_norm dx", gx, want_gx)
    assert_close("rms_norm dw", gw, want_gw)
