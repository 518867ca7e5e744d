"""The gated activation silu(x[:, :d]) * x[:, d:2d] against the fp64 oracle,
on decode and prefill shapes (MLP widths), both dtypes, the vectorised and the
element-wise kernels."""
import numpy as np
import pytest
import torch

import oracle
import rmsnorm_fwd_bwd_add_gb300 as rn
from parity import assert_close, f64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _library():
    from rmsnorm_fwd_bwd_add_gb300 import build
    build.build()


def _x(rows, d, dtype, seed, scale=3.0):
    gen = torch.Generator().manual_seed(seed)
    return (torch.randn(rows, 2 * d, generator=gen) * scale).to(dtype)


SHAPES = [(1, 14336), (4, 11008), (8, 4096), (300, 264), (2048, 14336), (7, 520),
          (5, 7), (33, 1001), (1, 1), (1000, 64)]


@pytest.mark.parametrize("rows,d", SHAPES, ids=["r%d_d%d" % s for s in SHAPES])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
def test_gated_silu_matches_oracle(rows, d, dtype):
    x = _x(rows, d, dtype, rows * 7 + d)
    out = rn.rmsnorm_gated_silu(x.to(DEV))
    assert out.shape == (rows, d) and out.dtype == dtype
    assert_close("gated silu", out, oracle.gated_silu(f64(x)))


def test_gated_silu_leading_dims_and_misaligned():
    x = _x(24, 4096, torch.bfloat16, 3).reshape(2, 3, 4, 8192)
    out = rn.rmsnorm_gated_silu(x.to(DEV))
    assert out.shape == (2, 3, 4, 4096)
    assert_close("gated silu 4-d", out.reshape(24, 4096), oracle.gated_silu(f64(x.reshape(24, 8192))))
    buf = torch.empty(24 * 8192 + 8, dtype=torch.bfloat16, device=DEV)
    xm = buf[1:1 + 24 * 8192].view(24, 8192)
    xm.copy_(x.reshape(24, 8192).to(DEV))
    assert xm.data_ptr() % 16 != 0
    assert_close("gated silu misaligned", rn.rmsnorm_gated_silu(xm),
                 oracle.gated_silu(f64(x.reshape(24, 8192))))


def test_gated_silu_extremes():
    # silu saturates: a -> +inf gives a*b, a -> -inf gives 0; no NaN from exp overflow
    a = torch.tensor([[80.0, -80.0, 0.0, 1e4, -1e4, 3.0]])
    b = torch.tensor([[2.0, 2.0, 5.0, 1.0, 1.0, -1.0]])
    x = torch.cat([a, b], dim=1).to(torch.bfloat16)
    out = rn.rmsnorm_gated_silu(x.to(DEV)).float().cpu()
    assert torch.all(torch.isfinite(out))
    want = oracle.gated_silu(f64(x))
    assert np.allclose(out.numpy(), want, rtol=4e-3, atol=1e-30)


def test_gated_silu_errors():
    x = torch.zeros(4, 16, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ValueError):
        rn.rmsnorm_gated_silu(torch.zeros(4, 15, dtype=torch.bfloat16, device=DEV))
    lib = rn._native.lib()
    # out overlapping x
    assert lib.rmsnorm_gated_silu(x.data_ptr(), x.data_ptr() + 32, 4, 8, 1, None) == 1
    assert lib.rmsnorm_gated_silu(x.data_ptr(), None, 4, 8, 1, None) == 1
    assert lib.rmsnorm_gated_silu(x.data_ptr(), x.data_ptr(), 0, 8, 1, None) == 0
