"""fp32 rows, rows a stride apart (slices of wider buffers) and the per-row
scale rstd that the forward writes and the VJP can take, against the fp64
oracle on every tier (staged sub-warp and CTA-per-row, direct, generic)."""
import numpy as np
import pytest
import torch

import oracle
import rmsnorm_fwd_bwd_add_gb300 as rn
from rmsnorm_fwd_bwd_add_gb300 import _native
from rmsnorm_fwd_bwd_add_gb300 import workloads as W
from parity import assert_close, assert_close_conditioned, f64, gx_term_magnitude

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
F32 = torch.float32


@pytest.fixture(scope="module", autouse=True)
def _library():
    from rmsnorm_fwd_bwd_add_gb300 import build
    build.build()
    yield
    assert rn.rmsnorm_device_status(clear=True) == 0


def _rstd_close(name, got, want):
    rel = np.abs(f64(got).reshape(-1) - want) / np.abs(want)
    assert rel.max() <= 1e-5, "%s: worst relative error %.3e" % (name, rel.max())


# (rows, D): staged sub-warp (64, 264), staged CTA per row (1024 .. 8192 in
# fp32), direct (rows <= 8, and fp32 rows past the staged limit), generic (odd D)
FP32_SHAPES = [(4096, 4096), (2048, 8192), (1000, 64), (777, 264), (300, 1024), (5, 4096),
               (1, 512), (64, 1001), (40, 12288), (9, 40000), (333, 1280), (129, 1792), (65, 2560),
               (33, 3584)]


@pytest.mark.parametrize("rows,D", FP32_SHAPES, ids=["r%d_d%d" % s for s in FP32_SHAPES])
def test_fp32_forward_and_rstd(rows, D):
    case = W.random_case(rows, D, F32, seed=rows + 7 * D, weight_bias=1.0, eps=1e-6)
    out, new_res, rstd = rn.rmsnorm_fwd_ex(case.x.to(DEV), case.w.to(DEV), case.eps,
                                           case.weight_bias, case.residual.to(DEV), rstd=True)
    want_out, _ = oracle.fwd(f64(case.x), f64(case.w), case.eps, case.weight_bias,
                             f64(case.residual))
    assert_close("fp32 out", out, want_out)
    # one IEEE fp32 add, rounded to nearest even, on both sides
    assert torch.equal(new_res.cpu(), case.x + case.residual)
    _rstd_close("fp32 rstd", rstd, oracle.rstd(f64(case.x), case.eps, f64(case.residual)))


@pytest.mark.parametrize("rows,D", FP32_SHAPES, ids=["r%d_d%d" % s for s in FP32_SHAPES])
def test_fp32_vjp(rows, D):
    case = W.random_case(rows, D, F32, seed=rows + 11 * D, weight_bias=0.0, eps=1e-5)
    x = case.x + case.residual
    gx, gw = rn.rmsnorm_vjp(x.to(DEV), case.w.to(DEV), case.g.to(DEV), case.eps)
    want_gx, want_gw = oracle.vjp(f64(x), f64(case.w), f64(case.g), case.eps)
    terms = gx_term_magnitude(x, case.w, case.g, case.eps, 0.0)
    assert_close_conditioned("fp32 gx", gx, want_gx, terms)
    assert_close("fp32 gw", gw, want_gw, F32)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, F32], ids=["bf16", "f16", "f32"])
@pytest.mark.parametrize("rows,D", [(2048, 4096), (600, 512), (6, 2048), (50, 1001)],
                         ids=["staged_cta", "staged_warp", "direct", "generic"])
def test_vjp_with_supplied_rstd(rows, D, dtype):
    case = W.random_case(rows, D, dtype, seed=rows * 3 + D, weight_bias=1.0, eps=1e-5)
    h = f64(case.x)
    rstd32 = oracle.rstd(h, case.eps).astype(np.float32)  # the scale as fp32 storage holds it
    g_res = W.random_case(rows, D, dtype, seed=rows + 1, residual=False).g
    gx, gw = rn.rmsnorm_vjp_ex(case.x.to(DEV), case.w.to(DEV), case.g.to(DEV), case.eps,
                               case.weight_bias, g_res.to(DEV),
                               rstd=torch.from_numpy(rstd32).to(DEV))
    want_gx, want_gw = oracle.vjp_rstd(h, f64(case.w), f64(case.g), rstd32.astype(np.float64),
                                       case.weight_bias)
    want_gx = want_gx + f64(g_res)
    terms = gx_term_magnitude(case.x, case.w, case.g, case.eps, case.weight_bias) + np.abs(f64(g_res))
    assert_close_conditioned("g_h with rstd", gx, want_gx, terms)
    assert_close("gw with rstd", gw, want_gw, F32)


def test_vjp_rstd_is_used_not_recomputed():
    """A scale twice the true one must change gx the way the formula says."""
    case = W.random_case(512, 2048, torch.bfloat16, seed=5, residual=False)
    h = f64(case.x)
    rstd2 = (2.0 * oracle.rstd(h, case.eps)).astype(np.float32)
    gx, gw = rn.rmsnorm_vjp_ex(case.x.to(DEV), case.w.to(DEV), case.g.to(DEV), case.eps,
                               rstd=torch.from_numpy(rstd2).to(DEV))
    want_gx, want_gw = oracle.vjp_rstd(h, f64(case.w), f64(case.g), rstd2.astype(np.float64))
    assert_close("gx with 2*rstd", gx, want_gx)
    assert_close("gw with 2*rstd", gw, want_gw, F32)


# Column offsets (elements) of x, residual, out, new_residual inside wider
# buffers: 16-byte aligned rows (staged/direct tiers) and misaligned ones.
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, F32], ids=["bf16", "f16", "f32"])
@pytest.mark.parametrize("rows,D,pad", [(3000, 4096, 64), (1500, 64, 16), (700, 1024, 32),
                                        (5, 2048, 8), (257, 512, 1)],
                         ids=["cta", "subwarp", "warp", "direct", "misaligned"])
def test_strided_forward_and_vjp(rows, D, pad, dtype):
    case = W.random_case(rows, D, dtype, seed=rows + D + pad, weight_bias=0.0, eps=1e-6)
    ld_in = 2 * D + pad
    src = torch.zeros(rows, ld_in, dtype=dtype)
    src[:, :D] = case.x
    src[:, D + pad:] = case.residual
    src = src.to(DEV)
    x, res = src[:, :D], src[:, D + pad:]
    ld_out = 2 * D + 2 * pad
    dst = torch.full((rows, ld_out), 7.0, dtype=dtype, device=DEV)
    out, new_res = dst[:, pad:pad + D], dst[:, pad + D + pad:]
    rn.rmsnorm_fwd_ex(x, case.w.to(DEV), case.eps, case.weight_bias, res, out=out,
                      new_residual=new_res)
    want_out, want_h = oracle.fwd(f64(case.x), f64(case.w), case.eps, case.weight_bias,
                                  f64(case.residual))
    assert_close("strided out", out, want_out)
    assert_close("strided new_residual", new_res, want_h)
    d = dst.cpu()
    assert torch.all(d[:, :pad] == 7.0) and torch.all(d[:, pad + D:2 * pad + D] == 7.0)

    # VJP of the fused op on the strided new_residual, with strided g and g_res
    gsrc = torch.zeros(rows, ld_in, dtype=dtype)
    gsrc[:, :D] = case.g
    gsrc[:, D + pad:] = case.x  # any values serve as the gradient of new_residual
    gsrc = gsrc.to(DEV)
    g, g_res = gsrc[:, :D], gsrc[:, D + pad:]
    gx_buf = torch.full((rows, ld_out), 7.0, dtype=dtype, device=DEV)
    gx = gx_buf[:, pad:pad + D]
    _, gw = rn.rmsnorm_vjp_ex(new_res, case.w.to(DEV), g, case.eps, case.weight_bias, g_res, gx=gx)
    h = new_res.cpu()
    want_gx, want_gw = oracle.fused_vjp(f64(h), f64(case.w), f64(case.g), case.eps,
                                        case.weight_bias, f64(case.x))
    terms = gx_term_magnitude(h, case.w, case.g, case.eps, case.weight_bias) + np.abs(f64(case.x))
    assert_close_conditioned("strided g_h", gx, want_gx, terms)
    assert_close("strided gw", gw, want_gw, F32)
    assert torch.all(gx_buf.cpu()[:, :pad] == 7.0)
    # the same problem dense gives bit-identical results (same plan, same order)
    gx2, gw2 = rn.rmsnorm_vjp_ex(new_res.contiguous(), case.w.to(DEV), g.contiguous(), case.eps,
                                 case.weight_bias, g_res.contiguous())
    if pad % 8 == 0:
        assert torch.equal(gx2, gx) and torch.equal(gw2.view(torch.int32), gw.view(torch.int32))


def test_strided_in_place_and_interleaved_halves():
    """out written over x and new_residual over residual, where x and residual
    are the two halves of one [rows, 2D] buffer."""
    rows, D = 1024, 2048
    case = W.random_case(rows, D, torch.bfloat16, seed=3)
    buf = torch.cat([case.x, case.residual], dim=1).to(DEV)
    x, res = buf[:, :D], buf[:, D:]
    rn.rmsnorm_fwd_ex(x, case.w.to(DEV), case.eps, 0.0, res, out=x, new_residual=res)
    want_out, want_h = oracle.fwd(f64(case.x), f64(case.w), case.eps, 0.0, f64(case.residual))
    assert_close("in-place out", x, want_out)
    assert_close("in-place new_residual", res, want_h)


def test_strided_argument_errors():
    rows, D = 16, 64
    buf = torch.zeros(rows, 2 * D, dtype=torch.bfloat16, device=DEV)
    w = torch.ones(D, dtype=torch.bfloat16, device=DEV)
    lib = _native.lib()
    x = buf.data_ptr()
    out = torch.empty(rows, D, dtype=torch.bfloat16, device=DEV)

    def fwd_ex(x_ptr, ld_x, out_ptr, ld_out):
        return lib.rmsnorm_fwd_ex(x_ptr, ld_x, None, 0, w.data_ptr(), 1e-6, 0.0, out_ptr, ld_out,
                                  None, 0, None, rows, D, 1, None)

    assert fwd_ex(x, D - 1, out.data_ptr(), D) == 1            # row stride < D
    assert fwd_ex(x, 2 * D, out.data_ptr(), D - 8) == 1        # output row stride < D
    assert fwd_ex(x, 2 * D, x + 2 * 8, 2 * D) == 1             # output overlaps x, shifted
    assert fwd_ex(x, 2 * D, x + 2 * D, 2 * D) == 0             # the other half: disjoint
    torch.cuda.synchronize()
    rstd_bad = buf[1, :2 * rows].view(torch.float32)  # in the span of x's rows
    assert lib.rmsnorm_fwd_ex(x + 2 * D, 2 * D, None, 0, w.data_ptr(), 1e-6, 0.0,
                              out.data_ptr(), D, None, 0, rstd_bad.data_ptr(), rows, D, 1,
                              None) == 1                        # rstd inside x's extent
    with pytest.raises(ValueError):
        rn.rmsnorm_fwd_ex(buf.t()[:D], w, 1e-6)                 # rows not contiguous


@pytest.mark.parametrize("dtype", [torch.bfloat16, F32], ids=["bf16", "f32"])
def test_autograd_on_strided_inputs(dtype):
    rows, D = 512, 1024
    case = W.random_case(rows, D, dtype, seed=17, weight_bias=1.0)
    big = torch.cat([case.x, case.residual], dim=1).to(DEV).requires_grad_()
    w = case.w.to(DEV).requires_grad_()
    out, new_res = rn.fused_add_rmsnorm(big[:, :D], big[:, D:], w, case.eps, 1.0)
    g_out = case.g.to(DEV)
    loss = (out.float() * g_out.float()).sum() + new_res.float().sum()
    gbig, gw = torch.autograd.grad(loss, (big, w))
    h = f64(new_res.detach())
    want_gh, want_gw = oracle.fused_vjp(h, f64(case.w), f64(case.g), case.eps, 1.0,
                                        np.ones((rows, D)))
    assert_close("autograd strided dx", gbig[:, :D], want_gh)
    assert torch.equal(gbig[:, :D], gbig[:, D:])
    assert_close("autograd strided dw", gw, want_gw)


def test_fp32_dispatch_and_gw_determinism():
    assert rn.rmsnorm_describe_dispatch("fwd", 4096, 4096, F32, True).startswith("staged")
    assert rn.rmsnorm_describe_dispatch("vjp", 4096, 8192, F32).startswith("staged")
    case = W.random_case(4096, 4096, F32, seed=9, residual=False)
    args = (case.x.to(DEV), case.w.to(DEV), case.g.to(DEV), case.eps)
    _, a = rn.rmsnorm_vjp(*args)
    _, b = rn.rmsnorm_vjp(*args)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_per_row_copy_fallback():
    """Strided sub-warp tiles without tensor maps (the path taken where the
    driver cannot make one): the strided and rstd cases above, rerun in a
    child process with the maps switched off."""
    import os
    import subprocess
    import sys
    env = dict(os.environ, RMSNORM_TUNE="tmap=0")
    r = subprocess.run([sys.executable, "-m", "pytest", __file__, "-q", "-x", "-p", "no:cacheprovider",
                        "-k", "test_strided_forward_and_vjp or test_vjp_with_supplied_rstd"],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
