"""Helpers for comparing the CUDA path with the fp64 oracle.

Tolerances (normwise relative error ||gpu - oracle||_2 / ||oracle||_2, over a
whole tensor and, for [rows, D] tensors, the worst single row):
  bf16 outputs 4e-3, fp16 outputs 1e-3, fp32 gw 1e-5, and 1e-5 for fp32
  outputs and rstd too: an fp32 result carries the sum of squares' error
  (at most about (terms per thread + tree depth) * 2^-24, ~2e-6 at D = 16384)
  plus a few roundings of the products, far below 1e-5.
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


U32 = 2.0 ** -24
# Half the spacing of the smallest subnormals: the absolute rounding error of
# an output that underflows.
HALF_SUBNORMAL = {torch.float16: 2.0 ** -25, torch.bfloat16: 2.0 ** -134,
                  torch.float32: 2.0 ** -150}


def gx_term_magnitude(x, w, g, eps, wb):
    """|r g w'| + |(r^3/D) h dot| elementwise: the size of the two terms whose
    difference is gx.  Their cancellation sets how many fp32 digits any
    evaluation of gx can keep (at D = 1 the terms agree to about
    log10(h^2/eps) digits)."""
    e = oracle.Oracle.scalar(eps)
    b = oracle.Oracle.scalar(wb)
    h = f64(x)
    u = f64(g) * (b + f64(w))[None, :]
    D = h.shape[1]
    r = 1.0 / np.sqrt(np.mean(h * h, axis=1) + e)
    dot = np.sum(u * h, axis=1)
    return np.abs(r[:, None] * u) + np.abs((r ** 3 / D * dot)[:, None] * h)


def assert_close_conditioned(name, got, want, terms, k=16.0):
    """Normwise check with the stated dtype tolerance plus the error that fp32
    cancellation of size `terms` and output underflow can cause: per row,
    ||err|| <= tol ||want|| + k u32 ||terms|| + sqrt(D) * half-subnormal.
    For the workload configurations the extra terms are far below tol."""
    tol = TOL[got.dtype]
    g = f64(got).reshape(-1, want.shape[-1])
    want = want.reshape(-1, want.shape[-1])
    terms = terms.reshape(-1, want.shape[-1])
    assert np.all(np.isfinite(g)), "%s: non-finite values in the GPU result" % name
    err = np.linalg.norm(g - want, axis=1)
    allow = (tol * np.linalg.norm(want, axis=1) + k * U32 * np.linalg.norm(terms, axis=1)
             + np.sqrt(want.shape[1]) * HALF_SUBNORMAL[got.dtype])
    bad = np.nonzero(err > allow)[0]
    assert bad.size == 0, "%s: row %d error %.3e > allowed %.3e" % (
        name, bad[0], err[bad[0]], allow[bad[0]])


def oracle_fwd(case, residual=True):
    res = case.residual if residual else None
    return oracle.fwd(f64(case.x), f64(case.w), case.eps, case.weight_bias,
                      None if res is None else f64(res))


def oracle_vjp(x_cpu: torch.Tensor, case):
    return oracle.vjp(f64(x_cpu), f64(case.w), f64(case.g), case.eps, case.weight_bias)
