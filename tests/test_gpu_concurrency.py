"""Calls captured in CUDA graphs and issued concurrently: the library's
stream-ordered scratch pool, its per-device set-up and its per-thread error
state under several streams and host threads."""
import threading

import pytest
import torch

import rmsnorm_fwd_bwd_add_gb300 as rn
from rmsnorm_fwd_bwd_add_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _library():
    from rmsnorm_fwd_bwd_add_gb300 import build
    build.build()
    yield
    assert rn.rmsnorm_device_status(clear=True) == 0


def _case(rows, D, seed):
    c = W.random_case(rows, D, torch.bfloat16, seed=seed)
    return c.x.to(DEV), c.residual.to(DEV), c.w.to(DEV), c.g.to(DEV), c.eps


def test_graph_capture_of_the_whole_step():
    """Forward, pooled VJP and fused VJP captured together and replayed give
    the eager results bit for bit (pool allocations inside the capture)."""
    x, res, w, g, eps = _case(3000, 4096, 1)
    eager = []
    out, nr = rn.rmsnorm_fwd(x, w, eps, 0.0, res)
    eager += [out.clone(), nr.clone()]
    gx, gw = rn.rmsnorm_vjp(nr, w, g, eps, 0.0)
    eager += [gx.clone(), gw.clone()]
    gh, gw2 = rn.rmsnorm_fused_vjp(nr, w, g, eps, 0.0, res)
    eager += [gh.clone(), gw2.clone()]
    torch.cuda.synchronize()

    outs = [torch.empty_like(t) for t in eager]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm up on the capture stream
        rn.rmsnorm_fwd(x, w, eps, 0.0, res, out=outs[0], new_residual=outs[1])
        rn.rmsnorm_vjp(outs[1], w, g, eps, 0.0, gx=outs[2], gw=outs[3])
        rn.rmsnorm_fused_vjp(outs[1], w, g, eps, 0.0, res, g_h=outs[4], gw=outs[5])
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        rn.rmsnorm_fwd(x, w, eps, 0.0, res, out=outs[0], new_residual=outs[1])
        rn.rmsnorm_vjp(outs[1], w, g, eps, 0.0, gx=outs[2], gw=outs[3])
        rn.rmsnorm_fused_vjp(outs[1], w, g, eps, 0.0, res, g_h=outs[4], gw=outs[5])
    for t in outs:
        t.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, outs):
        assert torch.equal(a.view(torch.int16) if a.dtype != torch.float32 else a.view(torch.int32),
                           b.view(torch.int16) if b.dtype != torch.float32 else b.view(torch.int32))


def test_concurrent_streams_and_threads():
    """Eight host threads, each on its own stream, run pooled VJPs and
    forwards at once; every result matches the same call made alone."""
    cases = [_case(600 + 97 * i, (512, 4096, 8192, 1000)[i % 4], 10 + i) for i in range(8)]
    ref = []
    for x, res, w, g, eps in cases:
        out, nr = rn.rmsnorm_fwd(x, w, eps, 0.0, res)
        gx, gw = rn.rmsnorm_vjp(nr, w, g, eps, 0.0)
        ref.append((out.clone(), gx.clone(), gw.clone()))
    torch.cuda.synchronize()
    results = [None] * len(cases)
    errors = []

    def work(i):
        try:
            x, res, w, g, eps = cases[i]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(5):
                    out, nr = rn.rmsnorm_fwd(x, w, eps, 0.0, res)
                    gx, gw = rn.rmsnorm_vjp(nr, w, g, eps, 0.0)
            s.synchronize()
            results[i] = (out, gx, gw)
        except Exception as e:  # surfaced below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for (o1, gx1, gw1), (o2, gx2, gw2) in zip(ref, results):
        assert torch.equal(o1, o2) and torch.equal(gx1, gx2)
        assert torch.equal(gw1.view(torch.int32), gw2.view(torch.int32))


def test_last_cuda_error_is_per_thread():
    """rmsnorm_last_cuda_error is thread-local: a new thread starts at 0
    whatever the calling thread has seen."""
    lib = rn._native.lib()
    seen = []

    def other():
        seen.append(lib.rmsnorm_last_cuda_error())

    t = threading.Thread(target=other)
    t.start()
    t.join()
    assert seen == [0]


def test_graph_capture_of_strided_calls_with_tensor_maps():
    """Rows a stride apart through the tensor-map path (sub-warp tiles) and the
    per-row scale, captured in a graph: the maps are encoded at capture time
    and the replays give the eager results bit for bit."""
    rows, D = 4000, 512
    c = W.random_case(rows, D, torch.bfloat16, seed=5)
    buf = torch.cat([c.x, c.residual], dim=1).to(DEV)
    x, res, w, g = buf[:, :D], buf[:, D:], c.w.to(DEV), c.g.to(DEV)
    obuf = torch.empty(rows, 2 * D, dtype=torch.bfloat16, device=DEV)

    def step(o):
        out, nr = o[0][:, :D], o[0][:, D:]
        rn.rmsnorm_fwd_ex(x, w, c.eps, 1.0, res, out=out, new_residual=nr, rstd=o[1])
        rn.rmsnorm_vjp_ex(nr, w, g, c.eps, 1.0, res, rstd=o[1], gx=o[2][:, :D], gw=o[3])

    eager = [obuf.clone(), torch.empty(rows, device=DEV),
             torch.empty(rows, 2 * D, dtype=torch.bfloat16, device=DEV),
             torch.empty(D, device=DEV)]
    step(eager)
    torch.cuda.synchronize()
    outs = [torch.empty_like(t) for t in eager]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(outs)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(outs)
    for t in outs:
        t.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(outs[0], eager[0])
    assert torch.equal(outs[1].view(torch.int32), eager[1].view(torch.int32))
    assert torch.equal(outs[2][:, :D], eager[2][:, :D])
    assert torch.equal(outs[3].view(torch.int32), eager[3].view(torch.int32))
