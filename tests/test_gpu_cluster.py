"""Rows longer than one CTA's shared-memory ring (more than 2048 16-byte
vectors): a thread-block cluster of 2, 4 or 8 CTAs takes each row, every CTA
streaming its own slice, and the slices' sums meet through distributed shared
memory.  The CUDA path is compared with the fp64 oracle on every element;
gw is checked bit for bit across runs and under CUDA-graph replay; a copy
that never arrives in one CTA of a cluster times out in every CTA of it
without hanging the GPU, and the next call is correct."""
import pytest
import torch

import oracle
import rmsnorm_fwd_bwd_add_gb300 as rn
from rmsnorm_fwd_bwd_add_gb300 import workloads as W
from parity import assert_close, f64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _library():
    from rmsnorm_fwd_bwd_add_gb300 import build
    build.build()
    rn.rmsnorm_debug_inject(-1, 0)
    yield
    assert rn.rmsnorm_device_status(clear=True) == 0, "a kernel reported a wait timeout"


def _plan(op, case, residual=False):
    return rn.rmsnorm_describe_dispatch(op, case.rows, case.D, case.dtype, residual)


def _check(case):
    x, res, w, g = (t.to(DEV) for t in (case.x, case.residual, case.w, case.g))
    for op, resid in (("fwd", True), ("fwd", False), ("vjp", False)):
        plan = _plan(op, case, resid)
        assert plan.startswith("cluster"), (op, plan)
    out, nr = rn.rmsnorm_fwd(x, w, case.eps, case.weight_bias, res)
    want_out, want_h = oracle.fwd(f64(case.x), f64(case.w), case.eps, case.weight_bias,
                                  f64(case.residual))
    assert_close(case.name + " out", out, want_out)
    assert_close(case.name + " new_residual", nr, want_h)
    out2, _ = rn.rmsnorm_fwd(x, w, case.eps, case.weight_bias)
    want2, _ = oracle.fwd(f64(case.x), f64(case.w), case.eps, case.weight_bias)
    assert_close(case.name + " out (no residual)", out2, want2)
    xr = torch.from_numpy(want_h).to(case.dtype)
    del out, nr, out2, want_out, want2
    xd = xr.to(DEV)
    gx, gw = rn.rmsnorm_vjp(xd, w, g, case.eps, case.weight_bias)
    want_gx, want_gw = oracle.vjp(f64(xr), f64(case.w), f64(case.g), case.eps, case.weight_bias)
    assert_close(case.name + " gx", gx, want_gx)
    assert_close(case.name + " gw", gw, want_gw, torch.float32)
    for _ in range(2):
        gw2 = rn.rmsnorm_vjp(xd, w, g, case.eps, case.weight_bias)[1]
        assert torch.equal(gw.view(torch.int32), gw2.view(torch.int32))
    gh, gwf = rn.rmsnorm_fused_vjp(xd, w, g, case.eps, case.weight_bias, res)
    want_gh, want_gwf = oracle.fused_vjp(f64(xr), f64(case.w), f64(case.g), case.eps,
                                         case.weight_bias, f64(case.residual))
    assert_close(case.name + " g_h", gh, want_gh)
    assert_close(case.name + " fused gw", gwf, want_gwf, torch.float32)


@pytest.mark.parametrize("rows,D,dtype", [
    (2000, 40000, torch.bfloat16),   # 5000 vectors a row
    (512, 65536, torch.bfloat16),    # 8192 vectors: the widest cluster VJP
    (300, 16392, torch.bfloat16),    # 2049 vectors: slices that do not divide the row
    (400, 40008, torch.bfloat16),    # 5001 vectors: the forward's clusters too
    (1000, 32768, torch.float16),
    (777, 20008, torch.float16),
    (3000, 12000, torch.float32),    # fp32: 3000 vectors
    (99, 65536, torch.float32),      # 16384 vectors: eight slices of 2048, three stages
], ids=lambda v: str(v).replace("torch.", ""))
def test_long_rows(rows, D, dtype):
    case = W.random_case(rows, D, dtype, seed=rows + D, weight_bias=0.0, eps=1e-6)
    case.name = "cluster_r%d_d%d" % (rows, D)
    _check(case)


@pytest.mark.parametrize("rows,D,dtype", [(1200, 32768, torch.bfloat16), (1300, 16384, torch.float32)],
                         ids=lambda v: str(v).replace("torch.", ""))
def test_forward_takes_the_deeper_ring(rows, D, dtype):
    """Rows of 4096 vectors with a residual: clusters of two would leave a
    three-slice ring, so with at least 32 rows a cluster the forward runs in
    clusters of four (five stages) while the VJP keeps clusters of two."""
    case = W.random_case(rows, D, dtype, seed=rows + D, weight_bias=0.0, eps=1e-6)
    case.name = "deeper_r%d_d%d" % (rows, D)
    assert _plan("fwd", case, True).endswith(":cl4"), _plan("fwd", case, True)
    assert _plan("vjp", case).endswith(":cl2"), _plan("vjp", case)
    _check(case)


def test_cluster_gw_under_graph_replay():
    case = W.random_case(600, 24576, torch.bfloat16, seed=5, residual=False)
    x, w, g = (t.to(DEV) for t in (case.x, case.w, case.g))
    assert _plan("vjp", case).startswith("cluster")
    want = rn.rmsnorm_vjp(x, w, g, case.eps)[1].clone()
    ws = torch.empty(rn.rmsnorm_vjp_workspace_size(600, 24576, case.dtype), dtype=torch.uint8,
                     device=DEV)
    gx = torch.empty_like(x)
    gw = torch.empty(24576, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        rn.rmsnorm_vjp_ws(x, w, g, case.eps, workspace=ws, gx=gx, gw=gw)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        rn.rmsnorm_vjp_ws(x, w, g, case.eps, workspace=ws, gx=gx, gw=gw)
    gw.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(gw.view(torch.int32), want.view(torch.int32))


def test_cluster_wait_timeout_is_reported_and_context_survives():
    """One CTA's copy of one row never arrives (host-side hook, short wait
    budget): that CTA times out on its copy, the rest of its cluster on the
    row sums it never sends; all leave through the bounded exit handshake,
    the timeout bit is set, and the next call is correct."""
    case = W.random_case(400, 40000, torch.bfloat16, seed=9, residual=False)
    x, w, g = (t.to(DEV) for t in (case.x, case.w, case.g))
    plan = _plan("vjp", case)
    assert plan.startswith("cluster"), plan
    cl = int(plan.split(":cl")[1])
    clusters = int(plan.split(":grid")[1].split(":")[0]) // cl
    rn.rmsnorm_device_status(clear=True)
    # cluster 1's third row, in the cluster's second CTA
    rn.rmsnorm_debug_inject(drop_tile=(1 + 2 * clusters) * cl + 1, budget_cycles=2_000_000)
    try:
        rn.rmsnorm_vjp(x, w, g, case.eps)
        bits = rn.rmsnorm_device_status(clear=True)
    finally:
        rn.rmsnorm_debug_inject(-1, 0)
    assert bits & rn.DEVSTATUS_WAIT_TIMEOUT
    gx, gw = rn.rmsnorm_vjp(x, w, g, case.eps)
    want_gx, want_gw = oracle.vjp(f64(case.x), f64(case.w), f64(case.g), case.eps, 0.0)
    assert_close("after timeout gx", gx, want_gx)
    assert_close("after timeout gw", gw, want_gw, torch.float32)
    assert rn.rmsnorm_device_status(clear=True) == 0
