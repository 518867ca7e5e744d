"""Seeded synthetic inputs with the shapes and value distributions of the
workloads the pages describe.  Shared by the tests and the benchmark; holds no
arithmetic of the method itself (only random draws and casts).

Recipe: values are drawn in fp32 on the CPU with
``torch.Generator().manual_seed(1000 + 100 * config + case)`` and cast to the
working dtype; the oracle and the CUDA path read the same cast values.

Configurations (the numbering used throughout):
  1  RMSNorm fwd + VJP, rows 64, D 512, fp16; x, w, g ~ U(0,1); eps 1e-5;
     weight_bias 0; no residual.  The (256, 512] fp16 band that the MLX CUDA
     kernel got wrong ("chore(deps): report the CUDA RMSNorm small-axis
     regression upstream ...", The upstream problem).
  2  decode fused add-RMSNorm, bf16, rows {1, 4, 8} x D {2048, 4096, 8192};
     x, residual ~ N(0,1); (i) w ~ N(1, 0.02), weight_bias 0, or (ii)
     w ~ N(0, 0.02), weight_bias 1; eps 1e-6.  The microbenchmark grid of
     "Fused residual-add RMSNorm and fused RoPE + KV-append decode kernels",
     Performance validation.  g ~ N(0,1) for VJP parity at these sizes.
  3  VJP rows 8192, D 4096, fp16; x, w, g ~ U(0,1); eps 1e-5; weight_bias 0.
     The POC workload of "RMSNormVJP backward writes a full {n_rows, D}
     gw_temp intermediate".
  4  prefill fused add-RMSNorm fwd + VJP, bf16, rows 16384, D {4096, 8192};
     x, residual ~ N(0,1), w ~ N(1, 0.02), g ~ N(0,1); eps 1e-6;
     weight_bias 0; the VJP runs on new_residual.
  5  sweep rows 4096, D in SWEEP_D, fp16 and bf16; x ~ N(0,1) with
     round(1% of rows) scaled by 1e3 and as many by 1e-4 (rows picked by a
     seeded permutation); g ~ N(0,1); w ~ N(1, 0.02); eps 1e-6;
     weight_bias 0; no residual.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

SWEEP_D = (64, 128, 256, 264, 320, 384, 448, 512, 520, 576, 1024)
DECODE_ROWS = (1, 4, 8)
DECODE_D = (2048, 4096, 8192)
PREFILL_D = (4096, 8192)


@dataclass
class Case:
    config: int
    name: str
    rows: int
    D: int
    dtype: torch.dtype
    eps: float
    weight_bias: float
    x: torch.Tensor
    w: torch.Tensor
    residual: Optional[torch.Tensor] = None
    g: Optional[torch.Tensor] = None


def generator(config: int, case: int) -> torch.Generator:
    return torch.Generator().manual_seed(1000 + 100 * config + case)


def _uniform(gen, shape):
    return torch.rand(shape, generator=gen, dtype=torch.float32)


def _normal(gen, shape, mean=0.0, std=1.0):
    return torch.randn(shape, generator=gen, dtype=torch.float32) * std + mean


def config1(case: int = 0) -> Case:
    gen = generator(1, case)
    rows, D, dt = 64, 512, torch.float16
    x = _uniform(gen, (rows, D)).to(dt)
    w = _uniform(gen, (D,)).to(dt)
    g = _uniform(gen, (rows, D)).to(dt)
    return Case(1, "c1_r64_d512_f16", rows, D, dt, 1e-5, 0.0, x, w, None, g)


def config2(rows: int, D: int, gemma: bool) -> Case:
    case = DECODE_ROWS.index(rows) * 10 + DECODE_D.index(D) * 2 + int(gemma)
    gen = generator(2, case)
    dt = torch.bfloat16
    x = _normal(gen, (rows, D)).to(dt)
    res = _normal(gen, (rows, D)).to(dt)
    if gemma:
        w, wb = _normal(gen, (D,), 0.0, 0.02).to(dt), 1.0
    else:
        w, wb = _normal(gen, (D,), 1.0, 0.02).to(dt), 0.0
    g = _normal(gen, (rows, D)).to(dt)
    name = "c2_r%d_d%d_%s" % (rows, D, "wb1" if gemma else "wb0")
    return Case(2, name, rows, D, dt, 1e-6, wb, x, w, res, g)


def config3(rows: int = 8192, D: int = 4096) -> Case:
    gen = generator(3, 0)
    dt = torch.float16
    x = _uniform(gen, (rows, D)).to(dt)
    w = _uniform(gen, (D,)).to(dt)
    g = _uniform(gen, (rows, D)).to(dt)
    return Case(3, "c3_r%d_d%d_f16" % (rows, D), rows, D, dt, 1e-5, 0.0, x, w, None, g)


def config4(D: int, rows: int = 16384) -> Case:
    gen = generator(4, PREFILL_D.index(D) if D in PREFILL_D else D)
    dt = torch.bfloat16
    x = _normal(gen, (rows, D)).to(dt)
    res = _normal(gen, (rows, D)).to(dt)
    w = _normal(gen, (D,), 1.0, 0.02).to(dt)
    g = _normal(gen, (rows, D)).to(dt)
    return Case(4, "c4_r%d_d%d_bf16" % (rows, D), rows, D, dt, 1e-6, 0.0, x, w, res, g)


def config4_on_device(D: int, device, rows: int = 16384) -> Case:
    """Configuration 4 drawn directly on `device` with a seeded CUDA generator:
    the same distributions as config4() (whose CPU draws the tests use), for
    benchmarks that need the inputs only in device memory."""
    gen = torch.Generator(device=device).manual_seed(1000 + 100 * 4 + (PREFILL_D.index(D) if D in PREFILL_D else D))
    dt = torch.bfloat16

    def normal(shape, mean=0.0, std=1.0):
        return torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std + mean
    x = normal((rows, D)).to(dt)
    res = normal((rows, D)).to(dt)
    w = normal((D,), 1.0, 0.02).to(dt)
    g = normal((rows, D)).to(dt)
    return Case(4, "c4_r%d_d%d_bf16" % (rows, D), rows, D, dt, 1e-6, 0.0, x, w, res, g)


def outlier_rows(rows: int, gen: torch.Generator):
    """Indices of the rows scaled by 1e3 and by 1e-4: round(1% of rows) each,
    taken from one seeded permutation."""
    k = int(round(0.01 * rows))
    perm = torch.randperm(rows, generator=gen)
    return perm[:k], perm[k:2 * k]


def config5(D: int, dtype: torch.dtype, rows: int = 4096) -> Case:
    if D in SWEEP_D:
        case = SWEEP_D.index(D) * 2 + (1 if dtype == torch.bfloat16 else 0)
    else:
        case = D
    gen = generator(5, case)
    x = _normal(gen, (rows, D))
    big, small = outlier_rows(rows, gen)
    x[big] *= 1e3
    x[small] *= 1e-4
    w = _normal(gen, (D,), 1.0, 0.02)
    g = _normal(gen, (rows, D))
    tag = "bf16" if dtype == torch.bfloat16 else "f16"
    return Case(5, "c5_r%d_d%d_%s" % (rows, D, tag), rows, D, dtype, 1e-6, 0.0,
                x.to(dtype), w.to(dtype), None, g.to(dtype))


def random_case(rows: int, D: int, dtype: torch.dtype, seed: int, residual: bool = True,
                weight_bias: float = 0.0, eps: float = 1e-6, scale: float = 1.0) -> Case:
    """Generic N(0,1) case for edge-shape tests (config number 0)."""
    gen = torch.Generator().manual_seed(seed)
    x = (_normal(gen, (rows, D)) * scale).to(dtype)
    res = _normal(gen, (rows, D)).to(dtype) if residual else None
    w = _normal(gen, (D,), 1.0 - weight_bias, 0.1).to(dtype)
    g = _normal(gen, (rows, D)).to(dtype)
    return Case(0, "rand_r%d_d%d" % (rows, D), rows, D, dtype, eps, weight_bias, x, w, res, g)
