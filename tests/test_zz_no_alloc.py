"""rmsnorm_vjp_noalloc, the VJP entry point for callers that may not allocate
device memory (runtimes that reserve all memory up front, plugin hosts that
provide no allocator or workspace, loops that cannot absorb an allocation).
It runs the same kernels as rmsnorm_vjp with the gw partials in a fixed array
inside the library.  This file is collected last so that a run stopping at the
first failure has already run every other test; it passes alone in a fresh
process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_close, f64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = {torch.bfloat16: 4e-3, torch.float16: 1e-3, torch.float32: 1e-5}
CODE = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2}


def _rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.fixture(scope="module")
def lib():
    from rmsnorm_fwd_bwd_add_gb300 import _native, build
    build.build()
    return _native.lib()


def _call_noalloc(lib, x, w, g, eps, wb):
    rows, D = x.shape
    gx = torch.empty_like(x)
    gw = torch.empty(D, dtype=torch.float32, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    st = lib.rmsnorm_vjp_noalloc(x.data_ptr(), w.data_ptr(), g.data_ptr(), eps, wb,
                                 gx.data_ptr(), gw.data_ptr(), rows, D, CODE[x.dtype], stream)
    return st, gx, gw


def test_noalloc_matches_rmsnorm_vjp_on_two_calls_in_a_row(lib):
    import rmsnorm_fwd_bwd_add_gb300 as rn
    from rmsnorm_fwd_bwd_add_gb300 import workloads as W
    # Two different problems back to back: the second must not see anything
    # the first left in the shared array.
    for rows, D, dtype, seed in ((4096, 4096, torch.bfloat16, 11), (1000, 1024, torch.float16, 12),
                                 (3000, 8192, torch.float32, 13)):
        case = W.random_case(rows, D, dtype, seed=seed, residual=False, weight_bias=1.0)
        x, w, g = case.x.to(DEV), case.w.to(DEV), case.g.to(DEV)
        gx_ref, gw_ref = rn.rmsnorm_vjp(x, w, g, case.eps, case.weight_bias)
        st, gx, gw = _call_noalloc(lib, x, w, g, case.eps, case.weight_bias)
        assert st == 0, rn.rmsnorm_status_string(st)
        torch.cuda.synchronize()
        assert _rel(gx, gx_ref) <= TOL[dtype]
        assert _rel(gw, gw_ref) <= 1e-5


@pytest.mark.parametrize("rows,D,dtype", [(1, 4096, torch.bfloat16), (2500, 8192, torch.float32),
                                          (16384, 4100, torch.bfloat16)])
def test_noalloc_matches_the_oracle(lib, rows, D, dtype):
    """Against the fp64 oracle directly: a decode row (one CTA: its partial
    row is gw itself and the array is not touched), an fp32 problem, and rows
    off 16-byte boundaries (D = 4100)."""
    from rmsnorm_fwd_bwd_add_gb300 import workloads as W
    case = W.random_case(rows, D, dtype, seed=rows + D, residual=False, weight_bias=0.0)
    x, w, g = case.x.to(DEV), case.w.to(DEV), case.g.to(DEV)
    st, gx, gw = _call_noalloc(lib, x, w, g, case.eps, case.weight_bias)
    assert st == 0
    want_gx, want_gw = oracle.vjp(f64(case.x), f64(case.w), f64(case.g), case.eps, 0.0)
    assert_close("noalloc gx", gx, want_gx)
    assert_close("noalloc gw", gw, want_gw, torch.float32)


def test_noalloc_gw_bits_survive_other_calls(lib):
    """Three calls of one problem with calls of other sizes in between, which
    leave other contents in the shared array: gw has the same bits each time."""
    from rmsnorm_fwd_bwd_add_gb300 import workloads as W
    a = W.random_case(5000, 2048, torch.bfloat16, seed=31, residual=False)
    b = W.random_case(777, 16384, torch.bfloat16, seed=32, residual=False)
    xa, wa, ga = a.x.to(DEV), a.w.to(DEV), a.g.to(DEV)
    xb, wb, gb = b.x.to(DEV), b.w.to(DEV), b.g.to(DEV)
    bits = []
    for _ in range(3):
        st, _, gw = _call_noalloc(lib, xa, wa, ga, a.eps, 0.0)
        assert st == 0
        bits.append(gw.view(torch.int32).clone())
        assert _call_noalloc(lib, xb, wb, gb, b.eps, 0.0)[0] == 0
    torch.cuda.synchronize()
    assert torch.equal(bits[0], bits[1]) and torch.equal(bits[0], bits[2])


@pytest.mark.parametrize("D,dtype", [(131072, torch.bfloat16), (65536, torch.float32)])
def test_noalloc_longest_aligned_rows(lib, D, dtype):
    """The longest aligned rows the array admits (16384 vectors: clusters of
    eight CTAs, one partial row per cluster) run and match the oracle; rows one
    vector longer run on the element-at-a-time tier, whose partial rows do not
    fit, and are refused."""
    from rmsnorm_fwd_bwd_add_gb300 import workloads as W
    case = W.random_case(24, D, dtype, seed=D, residual=False, weight_bias=0.0)
    x, w, g = case.x.to(DEV), case.w.to(DEV), case.g.to(DEV)
    st, gx, gw = _call_noalloc(lib, x, w, g, case.eps, 0.0)
    assert st == 0, lib.rmsnorm_status_string(st)
    want_gx, want_gw = oracle.vjp(f64(case.x), f64(case.w), f64(case.g), case.eps, 0.0)
    assert_close("noalloc gx D=%d" % D, gx, want_gx)
    assert_close("noalloc gw D=%d" % D, gw, want_gw, torch.float32)
    D2 = D + 16 // x.element_size()
    x2 = torch.zeros(2000, D2, dtype=dtype, device=DEV)
    st, _, _ = _call_noalloc(lib, x2, torch.ones(D2, dtype=dtype, device=DEV), x2, 1e-6, 0.0)
    assert st == 2


def test_noalloc_refuses_problems_beyond_its_array(lib):
    from rmsnorm_fwd_bwd_add_gb300 import _native
    # Long rows whose tensors sit at different offsets from 16-byte
    # boundaries run on the element-at-a-time tier, one partial row of D
    # floats per CTA for up to two CTAs per SM: 300 x 40000 floats (48 MB)
    # is far more than the fixed array holds.
    rows, D = 2000, 40000
    buf = torch.randn(rows * D + 8, device=DEV).to(torch.bfloat16)
    x = buf[1:1 + rows * D].view(rows, D)        # one element past a boundary
    g = torch.randn(rows, D, device=DEV).to(torch.bfloat16)
    w = torch.ones(D, dtype=torch.bfloat16, device=DEV)
    assert x.data_ptr() % 16 != g.data_ptr() % 16
    st, gx, gw = _call_noalloc(lib, x, w, g, 1e-6, 0.0)
    assert st == 2  # RMSNORM_ERR_UNSUPPORTED, nothing enqueued
    assert lib.rmsnorm_status_string(st) == b"unsupported problem size"
    assert _native.VJP_NOALLOC_MAX_BYTES == 16 << 20


def test_noalloc_python_binding_is_bit_identical_to_rmsnorm_vjp():
    import rmsnorm_fwd_bwd_add_gb300 as rn
    from rmsnorm_fwd_bwd_add_gb300 import workloads as W
    case = W.random_case(2048, 2048, torch.bfloat16, seed=21, residual=False)
    x, w, g = case.x.to(DEV), case.w.to(DEV), case.g.to(DEV)
    gx_ref, gw_ref = rn.rmsnorm_vjp(x, w, g, case.eps)
    gx, gw = rn.rmsnorm_vjp_noalloc(x, w, g, case.eps)
    # the same plan and summation order: the same bits
    assert torch.equal(gx, gx_ref)
    assert torch.equal(gw.view(torch.int32), gw_ref.view(torch.int32))
    with pytest.raises(rn.RmsnormError) as e:
        rows, D = 2000, 40000
        buf = torch.randn(rows * D + 8, device=DEV).to(torch.bfloat16)
        xl = buf[1:1 + rows * D].view(rows, D)
        gl = torch.randn(rows, D, device=DEV).to(torch.bfloat16)
        rn.rmsnorm_vjp_noalloc(xl, torch.ones(D, dtype=torch.bfloat16, device=DEV), gl, 1e-6)
    assert e.value.status == 2
