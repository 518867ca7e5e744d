"""Seeded random problems across the whole dispatch space, each checked against
the fp64 oracle on every element: row lengths from 1 to 131072 (log-uniform,
half of them rounded to whole 16-byte vectors), 1 to 20000 rows (a quarter of
them decode-sized), fp16, bf16 and fp32, with and without a residual,
weight_bias 0 or 1, and the row tensors at a shared offset from a 16-byte
boundary or at different offsets.  The forward (out, new_residual), the VJP
(gx, gw; gw bit for bit on a second call) and the two-output VJP run on every
problem.  A second set draws rows a stride apart (each tensor a slice of a
wider buffer, at its own padding) through the general entry points, with
the per-row scale written by the forward and supplied to the VJP on some
draws.  A third set draws the gated activation's shapes and offsets.  The
fixed edge lists elsewhere pin the tier boundaries; these draws land between
them."""
import numpy as np
import pytest
import torch

import oracle
import rmsnorm_fwd_bwd_add_gb300 as rn
from rmsnorm_fwd_bwd_add_gb300 import workloads as W
from parity import assert_close, assert_close_conditioned, f64, gx_term_magnitude

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
MAX_ELEMS = 1 << 22  # rows x D per problem: the oracle finishes each in well under a second


def _draw(i):
    rng = np.random.RandomState(9000 + i)
    dtype = [torch.bfloat16, torch.float16, torch.float32][rng.randint(3)]
    es = torch.empty(0, dtype=dtype).element_size()
    dmax = 131072 if es == 2 else 65536
    D = int(np.exp(rng.uniform(0.0, np.log(dmax))))
    if rng.rand() < 0.5:  # whole 16-byte vectors
        per = 16 // es
        D = max(per, D - D % per)
    D = max(1, min(D, dmax))
    if rng.rand() < 0.25:
        rows = int(rng.randint(1, 9))
    else:
        rows = int(np.exp(rng.uniform(np.log(9), np.log(20000))))
    rows = max(1, min(rows, MAX_ELEMS // D))
    u = rng.rand()
    offsets = (0, 0) if u < 0.6 else (1, 1) if u < 0.75 else (3, 3) if u < 0.9 else (1, 2)
    return dict(rows=rows, D=D, dtype=dtype, residual=bool(rng.rand() < 0.75),
                wb=float(rng.randint(2)), eps=float([1e-5, 1e-6][rng.randint(2)]),
                off=offsets, seed=int(rng.randint(1 << 30)))


DRAWS = [_draw(i) for i in range(128)]


def _ids(d):
    return "r%d_d%d_%s_off%d%d%s" % (d["rows"], d["D"], str(d["dtype"])[6:], d["off"][0],
                                    d["off"][1], "_res" if d["residual"] else "")


@pytest.fixture(scope="module", autouse=True)
def _library():
    from rmsnorm_fwd_bwd_add_gb300 import build
    build.build()
    rn.rmsnorm_debug_inject(-1, 0)
    yield
    assert rn.rmsnorm_device_status(clear=True) == 0, "a kernel reported a wait timeout"


def _at(t, off):
    """t's values in device memory `off` elements past a 16-byte boundary."""
    buf = torch.empty(t.numel() + 16, dtype=t.dtype, device=DEV)
    v = buf[off:off + t.numel()].view(t.shape)
    v.copy_(t.to(DEV))
    return v


def _empty_at(shape, dtype, off):
    n = int(np.prod(shape))
    buf = torch.full((n + 16,), float("nan"), dtype=dtype, device=DEV)
    return buf[off:off + n].view(shape)


@pytest.mark.parametrize("d", DRAWS, ids=[_ids(d) for d in DRAWS])
def test_random_problem(d):
    rows, D, dt, (o1, o2) = d["rows"], d["D"], d["dtype"], d["off"]
    case = W.random_case(rows, D, dt, seed=d["seed"], residual=True, weight_bias=d["wb"],
                         eps=d["eps"])
    case.name = _ids(d)
    x, g = _at(case.x, o1), _at(case.g, o1)
    res = _at(case.residual, o2) if d["residual"] else None
    w = _at(case.w, 0)
    out = _empty_at((rows, D), dt, o1)
    nr = _empty_at((rows, D), dt, o2) if d["residual"] else None
    rn.rmsnorm_fwd(x, w, case.eps, case.weight_bias, res, out=out, new_residual=nr)
    want_out, want_h = oracle.fwd(f64(case.x), f64(case.w), case.eps, case.weight_bias,
                                  f64(case.residual) if d["residual"] else None)
    assert_close(case.name + " out", out, want_out)
    if d["residual"]:
        assert_close(case.name + " new_residual", nr, want_h)
    # the VJP's input: the exact h rounded on the CPU, or x itself
    xr = torch.from_numpy(want_h).to(dt) if d["residual"] else case.x
    del out, nr, want_out, want_h
    xd = _at(xr, o1)
    gx = _empty_at((rows, D), dt, o1)
    _, gw = rn.rmsnorm_vjp(xd, w, g, case.eps, case.weight_bias, gx=gx)
    want_gx, want_gw = oracle.vjp(f64(xr), f64(case.w), f64(case.g), case.eps, case.weight_bias)
    terms = gx_term_magnitude(xr, case.w, case.g, case.eps, case.weight_bias)
    assert_close_conditioned(case.name + " gx", gx, want_gx, terms)
    assert_close(case.name + " gw", gw, want_gw, torch.float32)
    gw2 = rn.rmsnorm_vjp(xd, w, g, case.eps, case.weight_bias, gx=gx)[1]
    assert torch.equal(gw.view(torch.int32), gw2.view(torch.int32))
    gres = _at(case.residual, o2)
    gh = _empty_at((rows, D), dt, o1)
    _, gwf = rn.rmsnorm_fused_vjp(xd, w, g, case.eps, case.weight_bias, gres, g_h=gh)
    want_gh, want_gwf = oracle.fused_vjp(f64(xr), f64(case.w), f64(case.g), case.eps,
                                         case.weight_bias, f64(case.residual))
    assert_close_conditioned(case.name + " g_h", gh, want_gh, terms)
    assert_close(case.name + " fused gw", gwf, want_gwf, torch.float32)


def _draw_strided(i):
    rng = np.random.RandomState(7000 + i)
    dtype = [torch.bfloat16, torch.float16, torch.float32][rng.randint(3)]
    es = torch.empty(0, dtype=dtype).element_size()
    per = 16 // es
    D = int(np.exp(rng.uniform(0.0, np.log(20000 if es == 2 else 10000))))
    if rng.rand() < 0.5:
        D = max(per, D - D % per)
    if rng.rand() < 0.2:
        rows = int(rng.randint(1, 9))
    else:
        rows = int(np.exp(rng.uniform(np.log(9), np.log(8000))))

    def pad():  # elements past D in each row of a tensor's buffer
        return int(per * rng.randint(0, 9)) if rng.rand() < 0.6 else int(rng.randint(1, 2 * per))
    pads = dict(x=pad(), res=pad(), out=pad(), nr=pad(), g=pad(), gres=pad(), gx=pad())
    rows = max(1, min(rows, MAX_ELEMS // (D + max(pads.values()))))
    return dict(rows=rows, D=D, dtype=dtype, pads=pads, rstd=bool(rng.rand() < 0.5),
                gres=bool(rng.rand() < 0.5), wb=float(rng.randint(2)),
                eps=float([1e-5, 1e-6][rng.randint(2)]), seed=int(rng.randint(1 << 30)))


STRIDED = [_draw_strided(i) for i in range(48)]


def _sids(d):
    return "r%d_d%d_%s_ld+%d%s%s" % (d["rows"], d["D"], str(d["dtype"])[6:], d["pads"]["x"],
                                     "_rstd" if d["rstd"] else "", "_gres" if d["gres"] else "")


def _strided(t, padding, fill=None):
    """t's rows as a [rows, D] view into a [rows, D + padding] buffer."""
    rows, D = t.shape
    buf = torch.full((rows, D + padding), 7.0 if fill is None else fill, dtype=t.dtype, device=DEV)
    v = buf[:, :D]
    v.copy_(t.to(DEV))
    return v, buf


@pytest.mark.parametrize("d", STRIDED, ids=[_sids(d) for d in STRIDED])
def test_random_strided_problem(d):
    rows, D, dt, pads = d["rows"], d["D"], d["dtype"], d["pads"]
    case = W.random_case(rows, D, dt, seed=d["seed"], residual=True, weight_bias=d["wb"],
                         eps=d["eps"])
    case.name = _sids(d)
    w = case.w.to(DEV)
    x, _ = _strided(case.x, pads["x"])
    res, _ = _strided(case.residual, pads["res"])
    out, out_buf = _strided(torch.zeros(rows, D, dtype=dt), pads["out"])
    nr, nr_buf = _strided(torch.zeros(rows, D, dtype=dt), pads["nr"])
    _, _, r = rn.rmsnorm_fwd_ex(x, w, case.eps, case.weight_bias, res, out=out, new_residual=nr,
                                rstd=True if d["rstd"] else None)
    want_out, want_h = oracle.fwd(f64(case.x), f64(case.w), case.eps, case.weight_bias,
                                  f64(case.residual))
    assert_close(case.name + " out", out, want_out)
    assert_close(case.name + " new_residual", nr, want_h)
    for buf in (out_buf, nr_buf):  # the padding is untouched
        assert torch.all(buf[:, D:] == 7.0)
    if d["rstd"]:
        want_r = oracle.rstd(f64(case.x), case.eps, f64(case.residual))
        assert_close(case.name + " rstd", r, want_r, torch.float32)
    # the VJP on the exact h rounded on the CPU, rows a stride apart
    xr = torch.from_numpy(want_h).to(dt)
    del out, nr, want_out
    xv, _ = _strided(xr, pads["x"])
    g, _ = _strided(case.g, pads["g"])
    gres, _ = _strided(case.residual, pads["gres"]) if d["gres"] else (None, None)
    gx, gx_buf = _strided(torch.zeros(rows, D, dtype=dt), pads["gx"])
    rstd32 = oracle.rstd(f64(xr), case.eps).astype(np.float32) if d["rstd"] else None
    _, gw = rn.rmsnorm_vjp_ex(xv, w, g, case.eps, case.weight_bias, gres, gx=gx,
                              rstd=torch.from_numpy(rstd32).to(DEV) if d["rstd"] else None)
    if d["rstd"]:
        want_gx, want_gw = oracle.vjp_rstd(f64(xr), f64(case.w), f64(case.g),
                                           rstd32.astype(np.float64), case.weight_bias)
    else:
        want_gx, want_gw = oracle.vjp(f64(xr), f64(case.w), f64(case.g), case.eps,
                                      case.weight_bias)
    terms = gx_term_magnitude(xr, case.w, case.g, case.eps, case.weight_bias)
    if d["gres"]:
        want_gx = want_gx + f64(case.residual)
        terms = terms + np.abs(f64(case.residual))
    assert_close_conditioned(case.name + " gx", gx, want_gx, terms)
    assert_close(case.name + " gw", gw, want_gw, torch.float32)
    assert torch.all(gx_buf[:, D:] == 7.0)


def _draw_gated(i):
    rng = np.random.RandomState(5000 + i)
    dtype = [torch.bfloat16, torch.float16][rng.randint(2)]
    d = int(np.exp(rng.uniform(0.0, np.log(16384))))
    if rng.rand() < 0.5:
        d = max(8, d - d % 8)
    rows = int(np.exp(rng.uniform(0.0, np.log(5000))))
    rows = max(1, min(rows, MAX_ELEMS // (2 * d)))
    return dict(rows=rows, d=d, dtype=dtype, off=int([0, 0, 1, 3][rng.randint(4)]),
                seed=int(rng.randint(1 << 30)))


GATED = [_draw_gated(i) for i in range(24)]


@pytest.mark.parametrize("d", GATED, ids=["r%d_d%d_%s_off%d" % (g["rows"], g["d"],
                                                                  str(g["dtype"])[6:], g["off"])
                                          for g in GATED])
def test_random_gated_problem(d):
    gen = torch.Generator().manual_seed(d["seed"])
    x = (torch.randn(d["rows"], 2 * d["d"], generator=gen) * 3.0).to(d["dtype"])
    xd = _at(x, d["off"])
    out = rn.rmsnorm_gated_silu(xd)
    assert out.shape == (d["rows"], d["d"])
    assert_close("gated r%d d%d" % (d["rows"], d["d"]), out, oracle.gated_silu(f64(x)))
