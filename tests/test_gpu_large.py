"""Maximum sizes: more than 2^31 elements per tensor (64-bit indexing in every
tier that takes such rows), the longest supported row (D = 2^24) and the first
unsupported one.  Inputs are drawn on the device from a seeded generator;
outputs are checked on sampled rows, which the oracle computes one by one
(rows are independent), and gw through a g that is zero outside those rows,
so that the oracle's sum over the sampled rows is the whole gw."""
import numpy as np
import pytest
import torch

import oracle
import rmsnorm_fwd_bwd_add_gb300 as rn
from parity import assert_close, f64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

ROWS_2G = (1 << 31) // 4096 + 5  # 524293 rows of 4096: 2^31 + 20480 elements


@pytest.fixture(scope="module", autouse=True)
def _library():
    from rmsnorm_fwd_bwd_add_gb300 import build
    build.build()
    yield
    torch.cuda.empty_cache()
    assert rn.rmsnorm_device_status(clear=True) == 0


def _sample_rows(rows):
    """First and last rows, and the rows around element offsets 2^30 and 2^31
    (for D = 4096)."""
    cand = [0, 1, 262143, 262144, 524287, 524288, 524289, rows - 2, rows - 1]
    return sorted({r for r in cand if 0 <= r < rows})


def _randn(shape, dtype, gen):
    return torch.randn(shape, device=DEV, generator=gen, dtype=torch.float32).to(dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_over_2g_elements(dtype):
    rows, D = ROWS_2G, 4096
    gen = torch.Generator(device=DEV).manual_seed(2031)
    x = _randn((rows, D), dtype, gen)
    res = _randn((rows, D), dtype, gen)
    w = (1.0 + 0.02 * torch.randn(D, device=DEV, generator=gen)).to(dtype)
    assert rn.rmsnorm_describe_dispatch("fwd", rows, D, dtype, True).startswith("staged")
    out, nr, rstd = rn.rmsnorm_fwd_ex(x, w, 1e-6, 0.0, res, rstd=True)
    pick = torch.tensor(_sample_rows(rows), device=DEV)
    xs, rs, ws = f64(x[pick]), f64(res[pick]), f64(w)
    want_out, want_h = oracle.fwd(xs, ws, 1e-6, 0.0, rs)
    assert_close("out, sampled rows", out[pick], want_out)
    assert_close("new_residual, sampled rows", nr[pick], want_h)
    rel = np.abs(f64(rstd[pick]) - oracle.rstd(xs, 1e-6, rs)) / oracle.rstd(xs, 1e-6, rs)
    assert rel.max() <= 1e-5
    del out, nr, res, rstd

    # VJP: g is zero outside the sampled rows, so gw is their sum alone
    g = torch.zeros_like(x)
    g[pick] = _randn((len(pick), D), dtype, gen)
    gx, gw = rn.rmsnorm_vjp(x, w, g, 1e-6)
    want_gx, want_gw = oracle.vjp(xs, ws, f64(g[pick]), 1e-6)
    assert_close("gx, sampled rows", gx[pick], want_gx)
    assert_close("gw", gw, want_gw, torch.float32)
    # rows with g = 0 have gx = 0 exactly (every term carries a factor of g)
    assert torch.count_nonzero(gx[:8192][g[:8192].abs().sum(1) == 0]).item() == 0
    del x, g, gx
    torch.cuda.empty_cache()


def test_over_2g_elements_strided():
    """Rows 2D apart: the element offsets of the last rows pass 2^32."""
    rows, D = ROWS_2G, 4096
    gen = torch.Generator(device=DEV).manual_seed(2032)
    buf = _randn((rows, 2 * D), torch.bfloat16, gen)
    w = (1.0 + 0.02 * torch.randn(D, device=DEV, generator=gen)).to(torch.bfloat16)
    x = buf[:, D:]
    obuf = torch.empty_like(buf)
    out = obuf[:, :D]
    rn.rmsnorm_fwd_ex(x, w, 1e-6, 1.0, out=out)
    pick = torch.tensor(_sample_rows(rows), device=DEV)
    want_out, _ = oracle.fwd(f64(x[pick]), f64(w), 1e-6, 1.0)
    assert_close("strided out, sampled rows", out[pick], want_out)
    del buf, obuf, x, out
    torch.cuda.empty_cache()


def test_longest_row():
    """D = 2^24 (the largest supported), three rows, fwd and VJP in full."""
    rows, D = 3, 1 << 24
    assert D == rn.MAX_D
    gen = torch.Generator(device=DEV).manual_seed(2033)
    x = _randn((rows, D), torch.bfloat16, gen)
    res = _randn((rows, D), torch.bfloat16, gen)
    g = _randn((rows, D), torch.bfloat16, gen)
    w = (1.0 + 0.02 * torch.randn(D, device=DEV, generator=gen)).to(torch.bfloat16)
    out, nr = rn.rmsnorm_fwd(x, w, 1e-6, 0.0, res)
    want_out, want_h = oracle.fwd(f64(x), f64(w), 1e-6, 0.0, f64(res))
    assert_close("D=2^24 out", out, want_out)
    assert_close("D=2^24 new_residual", nr, want_h)
    gx, gw = rn.rmsnorm_vjp(x, w, g, 1e-6)
    want_gx, want_gw = oracle.vjp(f64(x), f64(w), f64(g), 1e-6)
    assert_close("D=2^24 gx", gx, want_gx)
    assert_close("D=2^24 gw", gw, want_gw, torch.float32)


def test_row_past_the_limit_is_unsupported():
    D = (1 << 24) + 8
    lib = rn._native.lib()
    x = torch.zeros(1, 8, dtype=torch.bfloat16, device=DEV)  # never read: rejected first
    st = lib.rmsnorm_fwd(x.data_ptr(), None, x.data_ptr(), 1e-6, 0.0, x.data_ptr(), None, 1, D,
                         1, None)
    assert st == 2
    assert rn.rmsnorm_describe_dispatch("fwd", 1, D, torch.bfloat16) == "invalid"
