"""Helpers for comparing the CUDA path with the fp64 oracle.

Tolerances (normwise relative error ||gpu - oracle||_2 / ||oracle||_2, over a
whole tensor and, for [rows, D] tensors, the worst single row):
  bf16 outputs 4e-3, fp16 outputs 1e-3, fp32 gw 1e-5.
bf16 keeps 8 significant bits (unit roundoff 2^-8 = 3.9e-3) and fp16 11
(2^-11 = 4.9e-4); one correct rounding of an fp32 result that is itself within
a few fp32 ulps of the exact value stays inside these bounds, a second
rounding or a lost term does not.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

TOL = {torch.bfloat16: 4e-3, torch.float16: 1e-3, torch.float32: 1e-5}


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact widening of a (CPU or CUDA) tensor to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def normwise(got: np.ndarray, want: np.ndarray) -> float:
    den = float(np.linalg.norm(want))
    num = float(np.linalg.norm(got - want))
    if den == 0.0:
        return num
    return num / den


def rowwise_max(got: np.ndarray, want: np.ndarray) -> float:
    if got.ndim < 2:
        return normwise(got, want)
    got = got.reshape(-1, got.shape[-1])
    want = want.reshape(-1, want.shape[-1])
    den = np.linalg.norm(want, axis=1)
    num = np.linalg.norm(got - want, axis=1)
    rel = np.where(den > 0, num / np.where(den > 0, den, 1.0), num)
    return float(rel.max()) if rel.size else 0.0


def assert_close(name: str, got: torch.Tensor, want: np.ndarray, dtype=None) -> None:
    tol = TOL[dtype if dtype is not None else got.dtype]
    g = f64(got)
    assert np.all(np.isfinite(g)), "%s: non-finite values in the GPU result" % name
    e_all = normwise(g, want)
    e_row = rowwise_max(g, want)
    assert e_all <= tol and e_row <= tol, (
        "%s: normwise error %.3e, worst row %.3e > tol %.1e" % (name, e_all, e_row, tol))


def oracle_fwd(case, residual=True):
    res = case.residual if residual else None
    return oracle.fwd(f64(case.x), f64(case.w), case.eps, case.weight_bias,
                      None if res is None else f64(res))


def oracle_vjp(x_cpu: torch.Tensor, case):
    return oracle.vjp(f64(x_cpu), f64(case.w), f64(case.g), case.eps, case.weight_bias)
