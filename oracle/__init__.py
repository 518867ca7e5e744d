"""fp64 CPU oracle for the RMSNorm hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(``rmsnorm_fwd_bwd_add_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``rmsnorm_oracle.c`` (plain C, fp64, rows and columns in
ascending order).  This module only compiles that file with gcc, loads it with
ctypes and marshals numpy float64 arrays.

Parity status: every function here is pinned (closed forms, hand-derived worked
examples, invariants, central finite differences, mutation tests) by
``tests/test_oracle_pins.py`` and ``tests/test_oracle_mutants.py``.

Sources (web pages, by title and section):
  * "Fused residual-add RMSNorm and fused RoPE + KV-append decode kernels",
    Background (FusedAddRMSNorm bullet; two-output paragraph) -- the forward,
    and the two-output op whose full VJP fused_vjp computes.
  * "RMSNormVJP backward writes a full {n_rows, D} gw_temp intermediate",
    POC section (eager fp32 reference and the gradient check) -- the VJP.
  * "Fused residual-add RMSNorm and fused RoPE + KV-append decode kernels",
    Background, third bullet -- the gated activation silu(x[:d]) * x[d:2d];
    second bullet and Task item 3 -- rope on q and k with the KV-cache append.
  * The same two pages' rsqrt(mean(h^2) + eps) factor -- rstd, the per-row
    scale a forward can hand to the backward, and the VJP that takes it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "rmsnorm_oracle.c")
BUILD_DIR = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "librmsnorm_oracle.so")

# -ffp-contract=off: no fused multiply-add contraction, so x86 and Arm hosts
# round every operation the same way.  No -ffast-math: no reassociation.
CFLAGS = ["-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def compile_source(source: str, out_path: str) -> str:
    """Compile a C oracle source file into a shared library at ``out_path``."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + ".tmp%d" % os.getpid()
    cmd = ["gcc", *CFLAGS, "-o", tmp, source, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Compile the oracle library if it is missing or older than its source."""
    if (not force and os.path.exists(LIB_PATH)
            and os.path.getmtime(LIB_PATH) >= os.path.getmtime(SOURCE)):
        return LIB_PATH
    return compile_source(SOURCE, LIB_PATH)


_dp = ctypes.POINTER(ctypes.c_double)


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    lib.rmsnorm_oracle_fwd.argtypes = [_dp, _dp, _dp, ctypes.c_double, ctypes.c_double,
                                       _dp, _dp, ctypes.c_int64, ctypes.c_int64]
    lib.rmsnorm_oracle_fwd.restype = None
    lib.rmsnorm_oracle_vjp.argtypes = [_dp, _dp, _dp, ctypes.c_double, ctypes.c_double,
                                       _dp, _dp, ctypes.c_int64, ctypes.c_int64]
    lib.rmsnorm_oracle_vjp.restype = None
    lib.rmsnorm_oracle_fused_vjp.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_double, ctypes.c_double,
                                             _dp, _dp, ctypes.c_int64, ctypes.c_int64]
    lib.rmsnorm_oracle_fused_vjp.restype = None
    lib.rmsnorm_oracle_gated_silu.argtypes = [_dp, _dp, ctypes.c_int64, ctypes.c_int64]
    lib.rmsnorm_oracle_gated_silu.restype = None
    lib.rmsnorm_oracle_rstd.argtypes = [_dp, _dp, ctypes.c_double, _dp, ctypes.c_int64,
                                        ctypes.c_int64]
    lib.rmsnorm_oracle_rstd.restype = None
    lib.rmsnorm_oracle_vjp_rstd.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_double, _dp, _dp,
                                            ctypes.c_int64, ctypes.c_int64]
    lib.rmsnorm_oracle_vjp_rstd.restype = None
    _ip = ctypes.POINTER(ctypes.c_int64)
    lib.rmsnorm_oracle_rope_kv_append.argtypes = [_dp, _dp, _dp, _ip, _ip, _dp, _dp, _dp, _dp,
                                                  ctypes.c_double, ctypes.c_int, ctypes.c_int64,
                                                  ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
    lib.rmsnorm_oracle_rope_kv_append.restype = None
    return lib


class Oracle:
    """numpy front end over one compiled oracle library (the real one, or a
    deliberately broken copy in the mutation tests)."""

    def __init__(self, lib_path: str):
        self.lib_path = lib_path
        self._lib = _bind(ctypes.CDLL(lib_path))

    @staticmethod
    def _arr(a, shape=None) -> np.ndarray:
        a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
        if shape is not None and a.shape != shape:
            raise ValueError("expected shape %s, got %s" % (shape, a.shape))
        return a

    @staticmethod
    def _ptr(a):
        return None if a is None else a.ctypes.data_as(_dp)

    @staticmethod
    def scalar(v: float) -> float:
        """The library takes eps and weight_bias as fp32 scalars; the oracle
        uses exactly the float32-rounded value, widened to double."""
        return float(np.float32(v))

    def fwd(self, x, w, eps, weight_bias=0.0, residual=None):
        """Returns (out, new_residual) as float64 arrays of x's 2-D shape;
        new_residual is None when residual is None."""
        x = self._arr(x)
        rows, D = x.shape
        w = self._arr(w, (D,))
        res = None if residual is None else self._arr(residual, (rows, D))
        out = np.empty((rows, D), np.float64)
        new_res = None if res is None else np.empty((rows, D), np.float64)
        self._lib.rmsnorm_oracle_fwd(self._ptr(x), self._ptr(res), self._ptr(w),
                                     self.scalar(eps), self.scalar(weight_bias),
                                     self._ptr(out), self._ptr(new_res), rows, D)
        return out, new_res

    def vjp(self, x, w, g, eps, weight_bias=0.0):
        """Returns (gx, gw): gx of x's 2-D shape, gw of shape (D,)."""
        x = self._arr(x)
        rows, D = x.shape
        w = self._arr(w, (D,))
        g = self._arr(g, (rows, D))
        gx = np.empty((rows, D), np.float64)
        gw = np.empty((D,), np.float64)
        self._lib.rmsnorm_oracle_vjp(self._ptr(x), self._ptr(w), self._ptr(g),
                                     self.scalar(eps), self.scalar(weight_bias),
                                     self._ptr(gx), self._ptr(gw), rows, D)
        return gx, gw

    def rstd(self, x, eps, residual=None):
        """Per-row 1 / sqrt(mean(h^2) + eps) of h = x + residual (or x), shape
        (rows,)."""
        x = self._arr(x)
        rows, D = x.shape
        res = None if residual is None else self._arr(residual, (rows, D))
        out = np.empty((rows,), np.float64)
        self._lib.rmsnorm_oracle_rstd(self._ptr(x), self._ptr(res), self.scalar(eps),
                                      self._ptr(out), rows, D)
        return out

    def vjp_rstd(self, x, w, g, rstd, weight_bias=0.0):
        """The VJP with the per-row scale rstd (shape (rows,)) supplied instead
        of recomputed; returns (gx, gw)."""
        x = self._arr(x)
        rows, D = x.shape
        w = self._arr(w, (D,))
        g = self._arr(g, (rows, D))
        rstd = self._arr(rstd, (rows,))
        gx = np.empty((rows, D), np.float64)
        gw = np.empty((D,), np.float64)
        self._lib.rmsnorm_oracle_vjp_rstd(self._ptr(x), self._ptr(w), self._ptr(g),
                                          self._ptr(rstd), self.scalar(weight_bias),
                                          self._ptr(gx), self._ptr(gw), rows, D)
        return gx, gw

    def fused_vjp(self, h, w, g_out, eps, weight_bias=0.0, g_residual=None):
        """VJP of the two-output fused op at h = x + residual: returns (g_h, gw),
        g_h the gradient with respect to both x and residual."""
        h = self._arr(h)
        rows, D = h.shape
        w = self._arr(w, (D,))
        g_out = self._arr(g_out, (rows, D))
        g_res = None if g_residual is None else self._arr(g_residual, (rows, D))
        g_h = np.empty((rows, D), np.float64)
        gw = np.empty((D,), np.float64)
        self._lib.rmsnorm_oracle_fused_vjp(self._ptr(h), self._ptr(w), self._ptr(g_out),
                                           self._ptr(g_res), self.scalar(eps),
                                           self.scalar(weight_bias), self._ptr(g_h),
                                           self._ptr(gw), rows, D)
        return g_h, gw


    def gated_silu(self, x):
        """x: (rows, 2d) -> silu(x[:, :d]) * x[:, d:], shape (rows, d)."""
        x = self._arr(x)
        rows, two_d = x.shape
        if two_d % 2:
            raise ValueError("x must have an even number of columns")
        d = two_d // 2
        out = np.empty((rows, d), np.float64)
        self._lib.rmsnorm_oracle_gated_silu(self._ptr(x), self._ptr(out), rows, d)
        return out


    def rope_kv_append(self, q, k, v, positions, slots, k_cache, v_cache, base=10000.0,
                       interleaved=False, cos_sin=None):
        """Returns (q_out, k_cache', v_cache'); the given caches are copied,
        not modified.  q: (T, Hq, Dh); k, v: (T, Hkv, Dh); caches
        (num_slots, Hkv, Dh); cos_sin: optional (max_pos, Dh) table."""
        q = self._arr(q)
        T, Hq, Dh = q.shape
        k = self._arr(k)
        Hkv = k.shape[1]
        v = self._arr(v, k.shape)
        kc = np.array(k_cache, dtype=np.float64, copy=True, order="C")
        vc = np.array(v_cache, dtype=np.float64, copy=True, order="C")
        pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int64))
        sl = np.ascontiguousarray(np.asarray(slots, dtype=np.int64))
        assert pos.shape == (T,) and sl.shape == (T,)
        cs = None if cos_sin is None else self._arr(cos_sin)
        q_out = np.empty_like(q)
        ip = ctypes.POINTER(ctypes.c_int64)
        self._lib.rmsnorm_oracle_rope_kv_append(
            self._ptr(q), self._ptr(k), self._ptr(v), pos.ctypes.data_as(ip), sl.ctypes.data_as(ip),
            self._ptr(q_out), self._ptr(kc), self._ptr(vc), self._ptr(cs), self.scalar(base),
            1 if interleaved else 0, T, Hq, Hkv, Dh)
        return q_out, kc, vc


_ORACLE = None


def load() -> Oracle:
    """The oracle built from ``rmsnorm_oracle.c`` (compiled on first use)."""
    global _ORACLE
    if _ORACLE is None:
        _ORACLE = Oracle(build())
    return _ORACLE


def fwd(x, w, eps, weight_bias=0.0, residual=None):
    return load().fwd(x, w, eps, weight_bias, residual)


def vjp(x, w, g, eps, weight_bias=0.0):
    return load().vjp(x, w, g, eps, weight_bias)


def rstd(x, eps, residual=None):
    return load().rstd(x, eps, residual)


def vjp_rstd(x, w, g, rstd, weight_bias=0.0):
    return load().vjp_rstd(x, w, g, rstd, weight_bias)


def fused_vjp(h, w, g_out, eps, weight_bias=0.0, g_residual=None):
    return load().fused_vjp(h, w, g_out, eps, weight_bias, g_residual)


def gated_silu(x):
    return load().gated_silu(x)


def rope_kv_append(q, k, v, positions, slots, k_cache, v_cache, base=10000.0, interleaved=False,
                   cos_sin=None):
    return load().rope_kv_append(q, k, v, positions, slots, k_cache, v_cache, base, interleaved,
                                 cos_sin)
