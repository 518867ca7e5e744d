"""Rows that start off a 16-byte boundary: D * size not a multiple of 16
(every row at a different offset), or tensors whose bases all sit at the
same unaligned offset.  These take the staged kernels' shifted-rows
instances: each row copied as its 16-byte aligned superset, aligned vectors
in and out, the two edge vectors of a row masked.  The CUDA path is compared
with the fp64 oracle on every element, at the prefill row count (16384) and
at sizes that leave ragged tiles; gw is also checked bit for bit across runs.
The unaligned-row failure the pages report for MLX's rewritten kernel
("chore(deps): report the CUDA RMSNorm small-axis regression upstream ...",
The upstream problem) is the case this file guards."""
import pytest
import torch

import oracle
import rmsnorm_fwd_bwd_add_gb300 as rn
from rmsnorm_fwd_bwd_add_gb300 import workloads as W
from parity import assert_close, assert_close_conditioned, f64, gx_term_magnitude

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _library():
    from rmsnorm_fwd_bwd_add_gb300 import build
    build.build()
    rn.rmsnorm_debug_inject(-1, 0)
    yield
    assert rn.rmsnorm_device_status(clear=True) == 0, "a kernel reported a wait timeout"


def _at_offset(t, offset_elems):
    """t's values in device memory that starts `offset_elems` elements past a
    16-byte boundary (offset 0: a fresh aligned copy)."""
    t = t.to(DEV)
    buf = torch.empty(t.numel() + 16, dtype=t.dtype, device=DEV)
    v = buf[offset_elems:offset_elems + t.numel()].view(t.shape)
    v.copy_(t)
    return v


def _empty_at(shape, dtype, offset_elems):
    buf = torch.full((int(torch.tensor(shape).prod()) + 16,), float("nan"), dtype=dtype,
                     device=DEV)
    return buf[offset_elems:offset_elems + buf.numel() - 16].view(shape)


def _run_all(case, off, expect_shift=True, conditioned=False):
    """Forward with residual, VJP on the rounded exact h, and the two-output
    VJP, every row tensor at `off` elements past a 16-byte boundary."""
    rows, D, dt = case.rows, case.D, case.dtype
    x, res, g = (_at_offset(t, off) for t in (case.x, case.residual, case.g))
    w = _at_offset(case.w, 0)
    if expect_shift:
        plan = rn.rmsnorm_describe_dispatch("fwd", rows, D, dt, True, 2 if off else 1)
        assert plan.startswith("staged-shift"), plan
    out, nr = _empty_at((rows, D), dt, off), _empty_at((rows, D), dt, off)
    rn.rmsnorm_fwd(x, w, case.eps, case.weight_bias, res, out=out, new_residual=nr)
    want_out, want_h = oracle.fwd(f64(case.x), f64(case.w), case.eps, case.weight_bias,
                                  f64(case.residual))
    assert_close(case.name + " out", out, want_out)
    assert_close(case.name + " new_residual", nr, want_h)
    xr = torch.from_numpy(want_h).to(dt)  # the exact h, rounded on the CPU
    del want_out, want_h, out, nr
    xd = _at_offset(xr, off)
    gx = _empty_at((rows, D), dt, off)
    _, gw = rn.rmsnorm_vjp(xd, w, g, case.eps, case.weight_bias, gx=gx)
    want_gx, want_gw = oracle.vjp(f64(xr), f64(case.w), f64(case.g), case.eps, case.weight_bias)
    if conditioned:
        terms = gx_term_magnitude(xr, case.w, case.g, case.eps, case.weight_bias)
        assert_close_conditioned(case.name + " gx", gx, want_gx, terms)
    else:
        assert_close(case.name + " gx", gx, want_gx)
    assert_close(case.name + " gw", gw, want_gw, torch.float32)
    # the same VJP again: the same gw bits
    gw2 = rn.rmsnorm_vjp(xd, w, g, case.eps, case.weight_bias, gx=gx)[1]
    assert torch.equal(gw.view(torch.int32), gw2.view(torch.int32))
    # the two-output op's VJP, with the residual standing in for g_residual
    gh = _empty_at((rows, D), dt, off)
    _, gwf = rn.rmsnorm_fused_vjp(xd, w, g, case.eps, case.weight_bias, res, g_h=gh)
    want_gh, want_gwf = oracle.fused_vjp(f64(xr), f64(case.w), f64(case.g), case.eps,
                                         case.weight_bias, f64(case.residual))
    if conditioned:
        assert_close_conditioned(case.name + " g_h", gh, want_gh, terms)
    else:
        assert_close(case.name + " g_h", gh, want_gh)
    assert_close(case.name + " fused gw", gwf, want_gwf, torch.float32)


# D * 2 bytes not a multiple of 16: rows every 8 (odd D), 4 (D = 2 mod 4) or
# 2 (D = 4 mod 8) rows apart share an offset; CTA-per-row and sub-warp shapes.
@pytest.mark.parametrize("D", [4100, 4097, 4098, 1001, 8200 + 4, 2050])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
def test_ragged_d_prefill_rows(D, dtype):
    case = W.random_case(16384, D, dtype, seed=D + 17, weight_bias=0.0, eps=1e-6)
    case.name = "shift_r16384_d%d" % D
    _run_all(case, 0)


# Every tensor's base at the same unaligned offset (a slice of a bigger
# buffer), D * 2 a multiple of 16: all rows at that offset.
@pytest.mark.parametrize("off", [1, 3, 7])
def test_shared_unaligned_base_prefill(off):
    case = W.random_case(16384, 4096, torch.bfloat16, seed=off, weight_bias=0.0, eps=1e-6)
    case.name = "shift_base%d_r16384_d4096" % off
    _run_all(case, off)


# Small and odd shapes: sub-warp tiles (D <= 1024 vectors' worth), ragged
# last tiles, a row shorter than one vector, and both offsets at once.
SMALL = [(9, 7), (100, 9), (1000, 63), (4099, 257), (301, 255), (37, 1025), (257, 515),
         (2000, 3075), (99, 6147), (41, 12291)]


@pytest.mark.parametrize("rows,D", SMALL, ids=["r%d_d%d" % s for s in SMALL])
@pytest.mark.parametrize("off", [0, 5])
def test_small_and_odd(rows, D, off):
    case = W.random_case(rows, D, torch.bfloat16, seed=rows * 31 + D + off, weight_bias=0.5,
                         eps=1e-5)
    _run_all(case, off, conditioned=True)


@pytest.mark.parametrize("rows,D,off", [(16384, 2051, 0), (4099, 1027, 1), (3000, 4096, 1),
                                        (513, 9, 3)])
def test_fp32_rows_off_boundary(rows, D, off):
    """fp32 rows: D % 4 != 0, or bases one to three elements (4-12 bytes) off."""
    case = W.random_case(rows, D, torch.float32, seed=rows + D, weight_bias=0.0, eps=1e-6)
    _run_all(case, off, conditioned=True)


def test_mixed_offsets_take_the_generic_tier():
    """Tensors at different offsets cannot share one aligned frame: the
    element-at-a-time tier runs them, still against the oracle."""
    case = W.random_case(300, 4096, torch.bfloat16, seed=3, weight_bias=0.0)
    x, res = _at_offset(case.x, 1), _at_offset(case.residual, 2)
    w = _at_offset(case.w, 0)
    out, nr = rn.rmsnorm_fwd(x, w, case.eps, 0.0, res)
    want_out, want_h = oracle.fwd(f64(case.x), f64(case.w), case.eps, 0.0, f64(case.residual))
    assert_close("mixed out", out, want_out)
    assert_close("mixed new_residual", nr, want_h)


def test_in_place_shifted():
    """out = x and new_residual = residual on shifted rows (D = 4097)."""
    case = W.random_case(2049, 4097, torch.bfloat16, seed=11)
    x, res = _at_offset(case.x, 0), _at_offset(case.residual, 0)
    w = _at_offset(case.w, 0)
    rn.rmsnorm_fwd(x, w, case.eps, 0.0, res, out=x, new_residual=res)
    want_out, want_h = oracle.fwd(f64(case.x), f64(case.w), case.eps, 0.0, f64(case.residual))
    assert_close("in-place out", x, want_out)
    assert_close("in-place new_residual", res, want_h)
