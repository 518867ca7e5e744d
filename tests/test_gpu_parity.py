"""CUDA path vs the fp64 oracle, element by element, on the seeded workloads
(all five configurations at full size) and on edge shapes that walk every
dispatch tier, ragged tails and unaligned rows.  All calls go through the C
ABI (via the thin ctypes binding)."""
import numpy as np
import pytest
import torch

import oracle
import rmsnorm_fwd_bwd_add_gb300 as rn
from rmsnorm_fwd_bwd_add_gb300 import workloads as W
from parity import (assert_close, assert_close_conditioned, f64, gx_term_magnitude, oracle_fwd,
                    oracle_vjp)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _library():
    from rmsnorm_fwd_bwd_add_gb300 import build
    build.build()
    rn.rmsnorm_debug_inject(-1, 0)
    yield
    assert rn.rmsnorm_device_status(clear=True) == 0, "a kernel reported a wait timeout"


def _dev(t):
    return None if t is None else t.to(DEV)


def _unit_roundoff(dtype):
    return 2.0 ** -8 if dtype == torch.bfloat16 else 2.0 ** -11


def check_fwd(case, residual=True):
    res = case.residual if residual else None
    out, nr = rn.rmsnorm_fwd(_dev(case.x), _dev(case.w), case.eps, case.weight_bias, _dev(res))
    want_out, want_h = oracle_fwd(case, residual)
    assert_close(case.name + " out", out, want_out)
    if residual:
        assert_close(case.name + " new_residual", nr, want_h)
        # new_residual is h rounded once: within one unit roundoff of the exact sum.
        got = f64(nr)
        bound = (_unit_roundoff(case.dtype) + 2.0 ** -23) * np.abs(want_h) + 2.0 ** -24
        assert np.all(np.abs(got - want_h) <= bound), case.name + " new_residual not rounded once"
    else:
        assert nr is None
    return out, nr, want_h


def check_vjp(case, x_cpu, conditioned=False):
    """conditioned=False: the stated tolerances as they are (the workload
    configurations).  conditioned=True (edge shapes, e.g. D = 1): gx also gets
    the error that fp32 cancellation between its two terms allows."""
    gx, gw = rn.rmsnorm_vjp(_dev(x_cpu), _dev(case.w), _dev(case.g), case.eps, case.weight_bias)
    want_gx, want_gw = oracle_vjp(x_cpu, case)
    if conditioned:
        terms = gx_term_magnitude(x_cpu, case.w, case.g, case.eps, case.weight_bias)
        assert_close_conditioned(case.name + " gx", gx, want_gx, terms)
    else:
        assert_close(case.name + " gx", gx, want_gx)
    assert_close(case.name + " gw", gw, want_gw, torch.float32)
    return gx, gw


def rounded_h(want_h, dtype):
    """The oracle's exact x + residual, rounded to the working dtype on the CPU:
    the VJP input for the fused pipeline (never taken from the CUDA path)."""
    return torch.from_numpy(want_h).to(dtype)


def check_fwd_unfused(case, out, xr):
    """The fused forward normalises the unrounded fp32 sum h; the unfused graph
    (add, round, then normalise) normalises round(h).  The two differ by at most
    one rounding of h, so the fused output also meets the tolerance against
    the oracle run on round(h) without a residual (the secondary check of the
    fused op's reading)."""
    want, _ = oracle.fwd(f64(xr), f64(case.w), case.eps, case.weight_bias)
    assert_close(case.name + " out against the unfused graph", out, want)


# ---- the five configurations -------------------------------------------------

def test_config1_small_multiwarp_band():
    case = W.config1()
    assert rn.rmsnorm_describe_dispatch("fwd", case.rows, case.D, case.dtype).startswith("staged")
    check_fwd(case, residual=False)
    check_vjp(case, case.x)


@pytest.mark.parametrize("rows", W.DECODE_ROWS)
@pytest.mark.parametrize("D", W.DECODE_D)
@pytest.mark.parametrize("gemma", [False, True], ids=["wb0", "wb1"])
def test_config2_decode(rows, D, gemma):
    case = W.config2(rows, D, gemma)
    assert rn.rmsnorm_describe_dispatch("fwd", rows, D, case.dtype, True).startswith("direct")
    out, nr, want_h = check_fwd(case)
    xr = rounded_h(want_h, case.dtype)
    mismatch = (nr.cpu() != xr).sum().item()
    assert mismatch <= max(1, nr.numel() // 10000)
    check_fwd_unfused(case, out, xr)
    check_vjp(case, xr)


def test_config3_vjp_8192x4096_fp16():
    case = W.config3()
    assert rn.rmsnorm_describe_dispatch("vjp", case.rows, case.D, case.dtype).startswith("staged")
    check_vjp(case, case.x)
    check_fwd(case, residual=False)


@pytest.mark.parametrize("D", W.PREFILL_D)
def test_config4_prefill(D):
    case = W.config4(D)
    out, nr, want_h = check_fwd(case)
    xr = rounded_h(want_h, case.dtype)
    del want_h
    mismatch = (nr.cpu() != xr).sum().item()
    assert mismatch <= nr.numel() // 10000
    del nr
    check_fwd_unfused(case, out, xr)
    del out
    check_vjp(case, xr)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("D", W.SWEEP_D)
def test_config5_sweep(D, dtype):
    case = W.config5(D, dtype)
    check_fwd(case, residual=False)
    check_vjp(case, case.x)


# ---- edge shapes: every tier, ragged tails, maximum sizes ---------------------

EDGE = [
    # (rows, D): direct (rows <= 8), generic (a few rows off 16-byte
    # boundaries, rows too long for any vectorised tier), shifted rows (D % 8
    # != 0 with more than 8 rows), staged small-D (D <= 1024) and CTA-per-row
    # (1024 < D <= 16384), clusters (aligned rows of more than 2048 vectors),
    # with row counts that leave ragged last tiles and uneven CTA loads.
    (1, 1), (3, 7), (2, 9), (5, 255), (9, 257), (17, 263), (33, 1000),
    (1, 8), (8, 64), (9, 64), (1000, 64), (301, 128), (157, 256), (999, 264),
    (4099, 520), (613, 1024), (2, 1032), (311, 1032), (305, 2048), (307, 4104),
    (153, 8192), (7, 16384), (155, 16384), (9, 16392), (3, 32768), (11, 40000),
    (2, 1 << 20),
    # CTA-per-row configurations that fit rows of 3 * 2^k vectors exactly
    # (96, 192, 384 and 768 threads), at and just past their widths
    (301, 1536), (257, 3072), (263, 2056), (97, 6144), (131, 12288), (35, 8200),
    # ... and of 5 * 2^k and 7 * 2^k vectors (160, 224, 320 and 448 threads)
    (311, 2560), (229, 3584), (151, 5120), (93, 7168), (41, 10240), (39, 14336),
]


@pytest.mark.parametrize("rows,D", EDGE, ids=["r%d_d%d" % e for e in EDGE])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_edge_shapes(rows, D, dtype):
    case = W.random_case(rows, D, dtype, seed=rows * 7919 + D, weight_bias=0.5, eps=1e-5)
    _, _, want_h = check_fwd(case, residual=True)
    check_fwd(case, residual=False)
    check_vjp(case, rounded_h(want_h, dtype), conditioned=True)


@pytest.mark.parametrize("rows,D,dtype", [(2, 2048, torch.bfloat16), (3, 4096, torch.float16),
                                          (5, 8192, torch.bfloat16), (7, 16384, torch.bfloat16),
                                          (8, 1024, torch.float32)],
                         ids=lambda v: str(v).replace("torch.", ""))
def test_decode_vjp_as_one_cluster(rows, D, dtype):
    """A decode VJP of 2-8 rows runs as one cluster of its rows that sums gw
    itself (plan ":cl<rows>", one kernel): gx and gw against the oracle, gw
    bit for bit across calls, and the same result with gw off a 16-byte
    boundary (one scratch row, then the fixed-order stage 2 of that row)."""
    case = W.random_case(rows, D, dtype, seed=rows * 1000 + D, residual=False, weight_bias=1.0)
    plan = rn.rmsnorm_describe_dispatch("vjp", rows, D, dtype)
    assert plan.startswith("direct") and plan.endswith(":cl%d" % rows), plan
    x = _dev(case.x)
    gx, gw = check_vjp(case, case.x)
    gw2 = rn.rmsnorm_vjp(x, _dev(case.w), _dev(case.g), case.eps, case.weight_bias)[1]
    assert torch.equal(gw.view(torch.int32), gw2.view(torch.int32))
    buf = torch.empty(D + 8, dtype=torch.float32, device=DEV)
    gw_off = buf[1:1 + D]  # 4 bytes past a 16-byte boundary
    assert gw_off.data_ptr() % 16 != 0
    gx3 = torch.empty_like(x)
    rn.rmsnorm_vjp(x, _dev(case.w), _dev(case.g), case.eps, case.weight_bias, gx=gx3, gw=gw_off)
    assert torch.equal(gx3, gx)
    assert torch.equal(gw_off.view(torch.int32), gw.view(torch.int32))


def test_empty_rows():
    x = torch.empty(0, 64, dtype=torch.bfloat16, device=DEV)
    w = torch.ones(64, dtype=torch.bfloat16, device=DEV)
    out, nr = rn.rmsnorm_fwd(x, w, 1e-6, 0.0, x.clone())
    assert out.shape == (0, 64) and nr.shape == (0, 64)
    gw = torch.full((64,), float("nan"), device=DEV)
    gx, gw = rn.rmsnorm_vjp(x, w, x.clone(), 1e-6, 0.0, gw=gw)
    assert torch.all(gw == 0), "empty VJP must write gw = 0"


@pytest.mark.parametrize("D", [64, 2048, 8192, 1001])
def test_single_row_vjp_gw(D):
    """One row runs as one CTA: with gw 16-byte aligned its partial row is written into gw in
    place (no second kernel); with gw 4 bytes off the two-stage path runs.  The in-place result
    matches the oracle, and the two paths give gw bit for bit."""
    case = W.random_case(1, D, torch.bfloat16, seed=D, weight_bias=1.0, eps=1e-5)
    check_vjp(case, case.x, conditioned=True)  # gw freshly allocated: aligned, in place
    x, w, g = _dev(case.x), _dev(case.w), _dev(case.g)
    gws = []
    for off in (0, 1):
        buf = torch.full((D + 4,), float("nan"), dtype=torch.float32, device=DEV)
        gws.append(rn.rmsnorm_vjp(x, w, g, case.eps, case.weight_bias, gw=buf[off:off + D])[1])
    assert torch.equal(gws[0].view(torch.int32), gws[1].view(torch.int32))


def _offset_view(t, offset_elems=1):
    """Same values as t, stored one element past a 16-byte boundary."""
    buf = torch.empty(t.numel() + 8, dtype=t.dtype, device=DEV)
    v = buf[offset_elems:offset_elems + t.numel()].view(t.shape)
    v.copy_(t.to(DEV))
    return v


@pytest.mark.parametrize("D", [512, 4096])
def test_misaligned_pointers(D):
    case = W.random_case(300, D, torch.bfloat16, seed=D, weight_bias=1.0)
    x, res, w, g = (_offset_view(t) for t in (case.x, case.residual, case.w, case.g))
    assert x.data_ptr() % 16 != 0
    assert rn.rmsnorm_describe_dispatch("fwd", 300, D, case.dtype, True, False).startswith("generic")
    out, nr = rn.rmsnorm_fwd(x, w, case.eps, case.weight_bias, res)
    want_out, want_h = oracle_fwd(case)
    assert_close("misaligned out", out, want_out)
    assert_close("misaligned new_residual", nr, want_h)
    xr = rounded_h(want_h, case.dtype)
    gx, gw = rn.rmsnorm_vjp(_offset_view(xr), w, g, case.eps, case.weight_bias)
    want_gx, want_gw = oracle_vjp(xr, case)
    assert_close("misaligned gx", gx, want_gx)
    assert_close("misaligned gw", gw, want_gw, torch.float32)


@pytest.mark.parametrize("rows,D", [(4, 4096), (500, 512), (300, 8192), (37, 100)])
def test_in_place(rows, D):
    case = W.random_case(rows, D, torch.bfloat16, seed=rows + D)
    x, res, w, g = _dev(case.x), _dev(case.residual), _dev(case.w), _dev(case.g)
    want_out, want_h = oracle_fwd(case)
    rn.rmsnorm_fwd(x, w, case.eps, case.weight_bias, res, out=x, new_residual=res)
    assert_close("in-place out", x, want_out)
    assert_close("in-place new_residual", res, want_h)
    xr = rounded_h(want_h, case.dtype)
    want_gx, want_gw = oracle_vjp(xr, case)
    xd = xr.to(DEV)
    gx, gw = rn.rmsnorm_vjp(xd, w, g, case.eps, case.weight_bias, gx=g)
    assert gx.data_ptr() == g.data_ptr()
    assert_close("in-place gx", g, want_gx)
    assert_close("in-place gw", gw, want_gw, torch.float32)


# ---- determinism, canaries, the workspace entry point ---------------------

@pytest.mark.parametrize("rows,D", [(8192, 4096), (4096, 512), (5, 8192), (300, 1001)])
def test_gw_bitwise_deterministic(rows, D):
    case = W.random_case(rows, D, torch.bfloat16, seed=99, residual=False)
    x, w, g = _dev(case.x), _dev(case.w), _dev(case.g)
    runs = [rn.rmsnorm_vjp(x, w, g, case.eps, 0.0)[1].clone() for _ in range(3)]
    for r in runs[1:]:
        assert torch.equal(r.view(torch.int32), runs[0].view(torch.int32))
    # the same bits from a CUDA-graph replay
    ws = torch.empty(rn.rmsnorm_vjp_workspace_size(rows, D, case.dtype), dtype=torch.uint8,
                     device=DEV)
    gx = torch.empty_like(x)
    gw = torch.empty(D, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        rn.rmsnorm_vjp_ws(x, w, g, case.eps, 0.0, workspace=ws, gx=gx, gw=gw)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        rn.rmsnorm_vjp_ws(x, w, g, case.eps, 0.0, workspace=ws, gx=gx, gw=gw)
    gw.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(gw.view(torch.int32), runs[0].view(torch.int32))


def test_vjp_ws_matches_vjp():
    case = W.config3(rows=1000)
    x, w, g = _dev(case.x), _dev(case.w), _dev(case.g)
    gx1, gw1 = rn.rmsnorm_vjp(x, w, g, case.eps, 0.0)
    gx2, gw2 = rn.rmsnorm_vjp_ws(x, w, g, case.eps, 0.0)
    assert torch.equal(gx1, gx2)
    assert torch.equal(gw1.view(torch.int32), gw2.view(torch.int32))


GUARD = 4096


def _guarded(rows, D, dtype):
    nbytes = rows * D * 2
    buf = torch.full((nbytes + 2 * GUARD,), 0xA5, dtype=torch.uint8, device=DEV)
    t = buf[GUARD:GUARD + nbytes].view(dtype).view(rows, D)
    t.fill_(float("nan"))
    return buf, t


def _guards_intact(buf):
    return bool(torch.all(buf[:GUARD] == 0xA5)) and bool(torch.all(buf[-GUARD:] == 0xA5))


@pytest.mark.parametrize("rows,D", [(3, 8192), (301, 4096), (1001, 520), (77, 33), (129, 16384)])
def test_canaries(rows, D):
    case = W.random_case(rows, D, torch.float16, seed=5)
    bo, out = _guarded(rows, D, case.dtype)
    bn, nr = _guarded(rows, D, case.dtype)
    rn.rmsnorm_fwd(_dev(case.x), _dev(case.w), case.eps, 0.0, _dev(case.residual),
                   out=out, new_residual=nr)
    bg, gx = _guarded(rows, D, case.dtype)
    gwbuf = torch.full((D + 2 * GUARD // 4,), float("nan"), device=DEV)
    gw = gwbuf[GUARD // 4:GUARD // 4 + D]
    rn.rmsnorm_vjp(nr, _dev(case.w), _dev(case.g), case.eps, 0.0, gx=gx, gw=gw)
    torch.cuda.synchronize()
    for name, b, t in (("out", bo, out), ("new_residual", bn, nr), ("gx", bg, gx)):
        assert _guards_intact(b), name + ": guard zone overwritten"
        assert torch.all(torch.isfinite(t)), name + ": element left unwritten"
    assert torch.all(torch.isnan(gwbuf[:GUARD // 4])) and torch.all(torch.isnan(gwbuf[-GUARD // 4:]))
    assert torch.all(torch.isfinite(gw))


# ---- errors and the timeout path -------------------------------------------

def test_errors_are_statuses():
    x = torch.randn(16, 64, device=DEV).to(torch.bfloat16)
    w = torch.ones(64, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(rn.RmsnormError) as e:
        rn.rmsnorm_fwd(x, w, -1.0)
    assert e.value.status == 1
    with pytest.raises(rn.RmsnormError) as e:
        rn.rmsnorm_fwd(x, w, float("nan"))
    assert e.value.status == 1
    # out overlapping x without being x
    big = torch.randn(17 * 64, device=DEV).to(torch.bfloat16)
    xv = big[:16 * 64].view(16, 64)
    ov = big[64:17 * 64].view(16, 64)
    with pytest.raises(rn.RmsnormError) as e:
        rn.rmsnorm_fwd(xv, w, 1e-6, out=ov)
    assert e.value.status == 1
    # workspace too small (this shape needs one [D] fp32 partial row per CTA)
    xl = torch.randn(4096, 1024, device=DEV).to(torch.bfloat16)
    wl = torch.ones(1024, dtype=torch.bfloat16, device=DEV)
    assert rn.rmsnorm_vjp_workspace_size(4096, 1024, torch.bfloat16) > 256
    with pytest.raises(rn.RmsnormError) as e:
        rn.rmsnorm_vjp_ws(xl, wl, xl, 1e-6, workspace=torch.empty(256, dtype=torch.uint8, device=DEV))
    assert e.value.status == 1
    # null workspace through the C ABI
    st = rn._native.lib().rmsnorm_vjp_ws(xl.data_ptr(), wl.data_ptr(), xl.data_ptr(), 1e-6, 0.0,
                                         torch.empty_like(xl).data_ptr(),
                                         torch.empty(1024, device=DEV).data_ptr(), 4096, 1024, 1,
                                         None, 1 << 30, None)
    assert st == 1


def test_wait_timeout_is_reported_and_context_survives():
    case = W.random_case(2000, 4096, torch.bfloat16, seed=3)
    x, res, w = _dev(case.x), _dev(case.residual), _dev(case.w)
    assert rn.rmsnorm_describe_dispatch("fwd", 2000, 4096, case.dtype, True).startswith("staged")
    rn.rmsnorm_device_status(clear=True)
    rn.rmsnorm_debug_inject(drop_tile=0, budget_cycles=2_000_000)
    try:
        rn.rmsnorm_fwd(x, w, case.eps, 0.0, res)
        bits = rn.rmsnorm_device_status(clear=True)
    finally:
        rn.rmsnorm_debug_inject(-1, 0)
    assert bits & rn.DEVSTATUS_WAIT_TIMEOUT
    # the context is still usable and the next call is correct
    check_fwd(case)
    assert rn.rmsnorm_device_status(clear=True) == 0


def test_vjp_wait_timeout_is_reported_and_context_survives():
    """The CTA-per-row VJP's row loop has no CTA barrier: a tile whose copy
    never arrives (dropped by the host-side hook) times out in every warp of
    that CTA, the timeout bit is set, and the next call is correct."""
    case = W.random_case(2000, 4096, torch.bfloat16, seed=5, residual=False)
    x, w, g = _dev(case.x), _dev(case.w), _dev(case.g)
    plan = rn.rmsnorm_describe_dispatch("vjp", 2000, 4096, case.dtype)
    assert plan.startswith("staged") and ":g256:" in plan, plan
    grid = int(plan.split(":grid")[1].split(":")[0])
    rn.rmsnorm_device_status(clear=True)
    rn.rmsnorm_debug_inject(drop_tile=grid + 3, budget_cycles=2_000_000)  # CTA 3's second row
    try:
        rn.rmsnorm_vjp(x, w, g, case.eps, case.weight_bias)
        bits = rn.rmsnorm_device_status(clear=True)
    finally:
        rn.rmsnorm_debug_inject(-1, 0)
    assert bits & rn.DEVSTATUS_WAIT_TIMEOUT
    check_vjp(case, case.x)
    assert rn.rmsnorm_device_status(clear=True) == 0


def test_injected_scratch_allocation_failure():
    """A failed gw scratch allocation (made on the host by the test hook, the
    allocator is not called) returns RMSNORM_ERR_NO_MEMORY with nothing
    enqueued; the next call allocates normally and is correct."""
    case = W.random_case(3000, 2048, torch.bfloat16, seed=41, residual=False)
    x, w, g = _dev(case.x), _dev(case.w), _dev(case.g)
    assert rn.rmsnorm_describe_dispatch("vjp", case.rows, case.D, case.dtype).startswith("staged")
    gx = torch.full_like(x, float("nan"))
    gw = torch.full((case.D,), float("nan"), dtype=torch.float32, device=DEV)
    rn.rmsnorm_debug_fail_allocs(1)
    try:
        with pytest.raises(rn.RmsnormError) as e:
            rn.rmsnorm_vjp(x, w, g, case.eps, case.weight_bias, gx=gx, gw=gw)
    finally:
        rn.rmsnorm_debug_fail_allocs(0)
    assert e.value.status == 4  # RMSNORM_ERR_NO_MEMORY
    torch.cuda.synchronize()
    assert torch.isnan(gx).all() and torch.isnan(gw).all(), "the failed call enqueued work"
    # the hook is spent: the same call now runs and matches the oracle
    rn.rmsnorm_vjp(x, w, g, case.eps, case.weight_bias, gx=gx, gw=gw)
    want_gx, want_gw = oracle_vjp(case.x, case)
    assert_close(case.name + " gx", gx, want_gx)
    assert_close(case.name + " gw", gw, want_gw, torch.float32)
    # a VJP that needs no scratch (one row: gw written in place) ignores the hook
    one = W.random_case(1, 2048, torch.bfloat16, seed=42, residual=False)
    rn.rmsnorm_debug_fail_allocs(1)
    try:
        gx1, gw1 = rn.rmsnorm_vjp(_dev(one.x), _dev(one.w), _dev(one.g), one.eps)
    finally:
        rn.rmsnorm_debug_fail_allocs(0)
    want_gx1, want_gw1 = oracle_vjp(one.x, one)
    assert_close("one row gx", gx1, want_gx1)
    assert_close("one row gw", gw1, want_gw1, torch.float32)


def test_bound_calls_match_the_oracle():
    """rmsnorm_fwd_bind / rmsnorm_vjp_bind (tensors checked once, the call
    issued on every invocation) on a decode step: the same bits as the plain
    calls, checked against the oracle, after several invocations."""
    case = W.config2(8, 4096, True)
    x, res, w, g = _dev(case.x), _dev(case.residual), _dev(case.w), _dev(case.g)
    fwd = rn.rmsnorm_fwd_bind(x, w, case.eps, case.weight_bias, res)
    for _ in range(3):
        out, nr = fwd()
    ref_out, ref_nr = rn.rmsnorm_fwd(x, w, case.eps, case.weight_bias, res)
    assert torch.equal(out, ref_out) and torch.equal(nr, ref_nr)
    want_out, want_h = oracle_fwd(case)
    assert_close("bound out", out, want_out)
    xr = _dev(rounded_h(want_h, case.dtype))
    vjp = rn.rmsnorm_vjp_bind(xr, w, g, case.eps, case.weight_bias)
    for _ in range(3):
        gx, gw = vjp()
    ref_gx, ref_gw = rn.rmsnorm_vjp(xr, w, g, case.eps, case.weight_bias)
    assert torch.equal(gx, ref_gx) and torch.equal(gw.view(torch.int32), ref_gw.view(torch.int32))
    want_gx, want_gw = oracle_vjp(xr.cpu(), case)
    assert_close("bound gx", gx, want_gx)
    assert_close("bound gw", gw, want_gw, torch.float32)
    with pytest.raises(ValueError):
        rn.rmsnorm_fwd_bind(x.cpu(), w, case.eps)
