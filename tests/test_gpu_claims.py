"""Staged forwards whose CTAs take their tiles from counters at run time.

The results must match the fp64 oracle whichever CTA takes a row; a counter
set reused by consecutive launches (the library's test hook narrows the
cycle to one set) must be left at zero by every launch, including one whose
wait timed out; a forward recorded into a CUDA graph keeps its own set and
replays correctly; and forwards on two streams at once, each on its own set,
give the same bits as on one stream."""
import pytest
import torch

import oracle
import rmsnorm_fwd_bwd_add_gb300 as rn
from rmsnorm_fwd_bwd_add_gb300 import workloads as W
from parity import assert_close, f64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

# (rows, D, dtype, residual): the forwards whose rows are long enough to be
# claimed (one CTA per SM, at least 96 KB moved per row), with row counts
# that are not a multiple of the grid.
SHAPES = [
    (2000, 12288, torch.bfloat16, True),
    (333, 16384, torch.bfloat16, True),
    (701, 14336, torch.float16, True),
    (1500, 8192, torch.float32, True),
]


@pytest.fixture(scope="module", autouse=True)
def _library():
    from rmsnorm_fwd_bwd_add_gb300 import build
    build.build()
    rn.rmsnorm_debug_inject(-1, 0)
    yield
    rn.rmsnorm_debug_claim_counters(0)
    assert rn.rmsnorm_device_status(clear=True) == 0, "a kernel reported a wait timeout"


def _case(rows, D, dtype, residual, seed):
    case = W.random_case(rows, D, dtype, seed=seed, residual=residual, weight_bias=0.0, eps=1e-6)
    case.name = "claims_r%d_d%d" % (rows, D)
    plan = rn.rmsnorm_describe_dispatch("fwd", rows, D, dtype, residual)
    assert plan.startswith("staged:") and plan.endswith(":claim"), plan
    return case


def _run(case, stream=None):
    x = case.x.to(DEV)
    w = case.w.to(DEV)
    res = case.residual.to(DEV) if case.residual is not None else None
    with torch.cuda.stream(stream or torch.cuda.current_stream()):
        out, nr = rn.rmsnorm_fwd(x, w, case.eps, case.weight_bias, res)
    return out, nr


def _check(case, out, nr):
    want_out, want_h = oracle.fwd(f64(case.x), f64(case.w), case.eps, case.weight_bias,
                                  None if case.residual is None else f64(case.residual))
    assert_close(case.name + " out", out, want_out)
    if case.residual is not None:
        assert_close(case.name + " new_residual", nr, want_h)


@pytest.mark.parametrize("rows,D,dtype,residual", SHAPES,
                         ids=lambda v: str(v).replace("torch.", ""))
def test_claimed_tiles_match_the_oracle(rows, D, dtype, residual):
    case = _case(rows, D, dtype, residual, seed=rows + D)
    out, nr = _run(case)
    _check(case, out, nr)


def test_one_counter_set_is_left_at_zero_by_every_launch():
    """With one counter set for every launch, a launch that did not put it
    back to zero would make the next one skip rows."""
    cases = [_case(*s, seed=100 + i) for i, s in enumerate(SHAPES)]
    rn.rmsnorm_debug_claim_counters(1)
    try:
        for _ in range(2):
            for case in cases:
                out, nr = _run(case)
                _check(case, out, nr)
        # a launch whose wait times out still leaves the set at zero
        case = cases[0]
        x, w, res = case.x.to(DEV), case.w.to(DEV), case.residual.to(DEV)
        rn.rmsnorm_device_status(clear=True)
        rn.rmsnorm_debug_inject(drop_tile=7, budget_cycles=2_000_000)
        try:
            rn.rmsnorm_fwd(x, w, case.eps, case.weight_bias, res)
            bits = rn.rmsnorm_device_status(clear=True)
        finally:
            rn.rmsnorm_debug_inject(-1, 0)
        assert bits & rn.DEVSTATUS_WAIT_TIMEOUT
        for case in cases:
            out, nr = _run(case)
            _check(case, out, nr)
        assert rn.rmsnorm_device_status(clear=True) == 0
    finally:
        rn.rmsnorm_debug_claim_counters(0)


def test_short_rows_keep_fixed_rows():
    """Rows too short for a claim to pay keep the static round robin."""
    for rows, D, dtype, residual in ((16384, 4096, torch.bfloat16, True),
                                     (16384, 8192, torch.bfloat16, True),
                                     (8192, 4096, torch.float16, False),
                                     (9001, 256, torch.bfloat16, True)):
        plan = rn.rmsnorm_describe_dispatch("fwd", rows, D, dtype, residual)
        assert plan.startswith("staged") and not plan.endswith(":claim"), plan
    for op in ("vjp",):
        plan = rn.rmsnorm_describe_dispatch(op, 2000, 12288, torch.bfloat16, False)
        assert not plan.endswith(":claim"), plan  # gw's order needs fixed rows


def test_claimed_tiles_under_graph_replay():
    case = _case(2000, 12288, torch.bfloat16, True, seed=7)
    x = case.x.to(DEV)
    res = case.residual.to(DEV)
    w = case.w.to(DEV)
    out = torch.empty_like(x)
    nr = torch.empty_like(x)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        rn.rmsnorm_fwd(x, w, case.eps, 0.0, res, out=out, new_residual=nr)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        rn.rmsnorm_fwd(x, w, case.eps, 0.0, res, out=out, new_residual=nr)
    for seed in (11, 12, 13):
        nxt = W.random_case(2000, 12288, torch.bfloat16, seed=seed, weight_bias=0.0, eps=1e-6)
        nxt.w = case.w
        nxt.name = "graph replay %d" % seed
        x.copy_(nxt.x.to(DEV))
        res.copy_(nxt.residual.to(DEV))
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        _check(nxt, out, nr)


def test_two_streams_at_once_give_the_one_stream_bits():
    a = _case(2000, 12288, torch.bfloat16, True, seed=21)
    b = _case(1500, 8192, torch.float32, True, seed=22)
    want_a = _run(a)[0].clone()
    want_b = _run(b)[0].clone()
    torch.cuda.synchronize()
    xa, wa, ra = a.x.to(DEV), a.w.to(DEV), a.residual.to(DEV)
    xb, wb, rb = b.x.to(DEV), b.w.to(DEV), b.residual.to(DEV)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    outs_a, outs_b = [], []
    for _ in range(12):
        with torch.cuda.stream(s1):
            outs_a.append(rn.rmsnorm_fwd(xa, wa, a.eps, 0.0, ra)[0])
        with torch.cuda.stream(s2):
            outs_b.append(rn.rmsnorm_fwd(xb, wb, b.eps, 0.0, rb)[0])
    torch.cuda.synchronize()
    for o in outs_a:
        assert torch.equal(o, want_a)
    for o in outs_b:
        assert torch.equal(o, want_b)
