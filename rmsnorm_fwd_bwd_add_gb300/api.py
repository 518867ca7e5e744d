"""Python front end of the C ABI: same names, argument marshalling only.

Every function checks dtype, device, contiguity and shape, then passes raw
pointers and the current CUDA stream to librmsnorm_gb300.so.  All arithmetic
runs in the library's CUDA kernels; nothing here computes.

Tensors: x, residual, g are [..., D] fp16, bf16 or fp32 CUDA tensors,
contiguous (the *_ex functions also take rows a stride apart: a slice of a
wider buffer); w is [D] of the same dtype; gw and rstd are fp32.  Leading
dimensions are flattened into rows.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import torch

from . import _native

_DTYPES = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2}


def _dtype_code(t: torch.Tensor, allowed=(0, 1, 2)) -> int:
    code = _DTYPES.get(t.dtype)
    if code is None or code not in allowed:
        names = {0: "fp16", 1: "bf16", 2: "fp32"}
        raise TypeError("unsupported dtype %s (%s)" % (
            t.dtype, " or ".join(names[c] for c in allowed))) from None
    return code


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else (t.data_ptr() or None)


def _check_like(name: str, t: torch.Tensor, ref: torch.Tensor) -> None:
    if t.dtype != ref.dtype or t.device != ref.device:
        raise ValueError("%s must be %s on %s" % (name, ref.dtype, ref.device))
    if t.shape != ref.shape:
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(ref.shape), tuple(t.shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def _rows_d(x: torch.Tensor) -> Tuple[int, int]:
    if x.dim() < 1:
        raise ValueError("x must have at least one dimension")
    if not x.is_cuda:
        raise ValueError("tensors must be CUDA tensors (there is no CPU path)")
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    D = x.shape[-1]
    return (x.numel() // D if D else 0), D


# The current stream's raw handle without building a Stream object (a private
# torch entry point present in the supported versions; the public route is the
# fallback).
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(device: torch.device, stream) -> int:
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(device.index)
    return torch.cuda.current_stream(device).cuda_stream


class _OnDevice:
    """Makes `device` current for the C call (the library works on the current
    device), switching only when it is not already."""

    __slots__ = ("device", "prev")

    def __init__(self, device: torch.device):
        self.device = device
        self.prev = None

    def __enter__(self):
        cur = torch.cuda.current_device()
        if cur != self.device.index:
            self.prev = cur
            torch.cuda.set_device(self.device)
        return self

    def __exit__(self, *exc):
        if self.prev is not None:
            torch.cuda.set_device(self.prev)
        return False


def _rows_ld(name: str, t: torch.Tensor) -> Tuple[int, int, int]:
    """(rows, D, row stride in elements) of a [..., D] CUDA tensor whose rows
    are contiguous and whose leading dimensions flatten to one row stride."""
    if t.dim() < 1:
        raise ValueError("%s must have at least one dimension" % name)
    if not t.is_cuda:
        raise ValueError("tensors must be CUDA tensors (there is no CPU path)")
    D = t.shape[-1]
    rows = t.numel() // D if D else 0
    if D > 1 and t.stride(-1) != 1:
        raise ValueError("%s: the elements of a row must be contiguous" % name)
    lead = [(n, st) for n, st in zip(t.shape[:-1], t.stride()[:-1]) if n != 1]
    if rows <= 1 or not lead:
        return rows, D, D
    for (n0, st0), (n1, st1) in zip(lead, lead[1:]):
        if st0 != st1 * n1:
            raise ValueError("%s: leading dimensions do not flatten to one row stride" % name)
    if lead[-1][1] < D:
        raise ValueError("%s: rows overlap (row stride %d < D = %d)" % (name, lead[-1][1], D))
    return rows, D, lead[-1][1]


def rows_layout_ok(t: torch.Tensor) -> bool:
    """Whether the *_ex functions take t's layout as it is (contiguous rows,
    one row stride >= D); callers copy other tensors with .contiguous()."""
    try:
        _rows_ld("t", t)
    except ValueError:
        return False
    return True


def _check_rows_like(name: str, t: torch.Tensor, ref: torch.Tensor) -> int:
    """Checks dtype, device and shape against ref; returns t's row stride."""
    if t.dtype != ref.dtype or t.device != ref.device:
        raise ValueError("%s must be %s on %s" % (name, ref.dtype, ref.device))
    if t.shape != ref.shape:
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(ref.shape), tuple(t.shape)))
    return _rows_ld(name, t)[2]


def _check_w(w: torch.Tensor, x: torch.Tensor, D: int) -> None:
    if w.dtype != x.dtype or w.device != x.device or w.shape != (D,) or not w.is_contiguous():
        raise ValueError("w must be a contiguous [%d] %s tensor on %s" % (D, x.dtype, x.device))


# ---- the per-token entry points: one cheap pass of checks per tensor -------
# A decode step calls these once per layer and token, so their Python cost is
# kept to a few attribute reads per tensor: dtype by identity, the device as an
# index, the shape, contiguity.  The message of a failed check is built only
# when it fails.

_get_device = getattr(torch._C, "_cuda_getDevice", None)
_fns = {}


def _fn(name: str):
    """The C entry point `name`, bound once."""
    f = _fns.get(name)
    if f is None:
        f = _fns[name] = getattr(_native.lib(), name)
    return f


def _rows_dev(x: torch.Tensor):
    """(rows, D, device index, dtype code) of a contiguous [..., D] CUDA tensor."""
    dev = x.get_device()
    if dev < 0:
        raise ValueError("tensors must be CUDA tensors (there is no CPU path)")
    shape = x.shape
    if not shape:
        raise ValueError("x must have at least one dimension")
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    code = _DTYPES.get(x.dtype)
    if code is None:
        _dtype_code(x)  # raises with the message
    D = shape[-1]
    return (x.numel() // D if D else 0), D, dev, code


def _like(name: str, t: torch.Tensor, x: torch.Tensor, dev: int) -> None:
    if (t.dtype is not x.dtype or t.get_device() != dev or t.shape != x.shape
            or not t.is_contiguous()):
        _check_like(name, t, x)  # raises with the message
        raise ValueError("%s must be a contiguous %s tensor on cuda:%d" % (name, x.dtype, dev))


def _weight(w: torch.Tensor, x: torch.Tensor, D: int, dev: int) -> None:
    if (w.dtype is not x.dtype or w.get_device() != dev or w.dim() != 1 or w.shape[0] != D
            or not w.is_contiguous()):
        _check_w(w, x, D)
        raise ValueError("w must be a contiguous [%d] %s tensor on cuda:%d" % (D, x.dtype, dev))


def _gw(gw: Optional[torch.Tensor], D: int, dev: int) -> torch.Tensor:
    if gw is None:
        return torch.empty(D, dtype=torch.float32, device=torch.device("cuda", dev))
    if (gw.dtype is not torch.float32 or gw.get_device() != dev or gw.dim() != 1
            or gw.shape[0] != D or not gw.is_contiguous()):
        raise ValueError("gw must be a contiguous [%d] float32 tensor on cuda:%d" % (D, dev))
    return gw


def _call(dev: int, stream, fn, *args) -> int:
    """fn(*args, stream) with device `dev` current (switched only if needed)."""
    cur = _get_device() if _get_device is not None else torch.cuda.current_device()
    h = stream.cuda_stream if stream is not None else (
        _raw_stream(dev) if _raw_stream is not None else torch.cuda.current_stream(dev).cuda_stream)
    if cur == dev:
        return fn(*args, h)
    torch.cuda.set_device(dev)
    try:
        return fn(*args, h)
    finally:
        torch.cuda.set_device(cur)


def rmsnorm_fwd(x: torch.Tensor, w: torch.Tensor, eps: float, weight_bias: float = 0.0,
                residual: Optional[torch.Tensor] = None, *, out: Optional[torch.Tensor] = None,
                new_residual: Optional[torch.Tensor] = None, stream=None):
    """Fused residual-add RMSNorm forward.  Returns (out, new_residual);
    new_residual is None when residual is None.  Pass out=x or
    new_residual=residual to update in place."""
    rows, D, dev, code = _rows_dev(x)
    _weight(w, x, D, dev)
    if out is None:
        out = torch.empty_like(x)
    else:
        _like("out", out, x, dev)
    if residual is not None:
        _like("residual", residual, x, dev)
        if new_residual is None:
            new_residual = torch.empty_like(x)
        else:
            _like("new_residual", new_residual, x, dev)
        st = _call(dev, stream, _fn("rmsnorm_fwd"), x.data_ptr() or None,
                   residual.data_ptr() or None, w.data_ptr(), eps, weight_bias,
                   out.data_ptr() or None, new_residual.data_ptr() or None, rows, D, code)
    elif new_residual is not None:
        raise ValueError("new_residual given without residual")
    else:
        st = _call(dev, stream, _fn("rmsnorm_fwd"), x.data_ptr() or None, None, w.data_ptr(),
                   eps, weight_bias, out.data_ptr() or None, None, rows, D, code)
    if st:
        _native.check("rmsnorm_fwd", st)
    return out, new_residual


def rmsnorm_vjp(x: torch.Tensor, w: torch.Tensor, g: torch.Tensor, eps: float,
                weight_bias: float = 0.0, *, gx: Optional[torch.Tensor] = None,
                gw: Optional[torch.Tensor] = None, stream=None):
    """RMSNorm VJP.  Returns (gx, gw) with gw fp32, reduced across rows on the
    GPU.  The library takes its gw scratch from its own stream-ordered pool."""
    rows, D, dev, code = _rows_dev(x)
    _weight(w, x, D, dev)
    _like("g", g, x, dev)
    if gx is None:
        gx = torch.empty_like(x)
    else:
        _like("gx", gx, x, dev)
    gw = _gw(gw, D, dev)
    st = _call(dev, stream, _fn("rmsnorm_vjp"), x.data_ptr() or None, w.data_ptr(),
               g.data_ptr() or None, eps, weight_bias, gx.data_ptr() or None, gw.data_ptr(), rows,
               D, code)
    if st:
        _native.check("rmsnorm_vjp", st)
    return gx, gw


def rmsnorm_fused_vjp(h: torch.Tensor, w: torch.Tensor, g_out: torch.Tensor, eps: float,
                      weight_bias: float = 0.0, g_residual: Optional[torch.Tensor] = None, *,
                      g_h: Optional[torch.Tensor] = None, gw: Optional[torch.Tensor] = None,
                      stream=None):
    """VJP of the two-output fused op at h (its new_residual): returns
    (g_h, gw), g_h = VJP(h, g_out) + g_residual the gradient with respect to
    both x and residual."""
    rows, D, dev, code = _rows_dev(h)
    _weight(w, h, D, dev)
    _like("g_out", g_out, h, dev)
    if g_residual is not None:
        _like("g_residual", g_residual, h, dev)
    if g_h is None:
        g_h = torch.empty_like(h)
    else:
        _like("g_h", g_h, h, dev)
    gw = _gw(gw, D, dev)
    st = _call(dev, stream, _fn("rmsnorm_fused_vjp"), h.data_ptr() or None, w.data_ptr(),
               g_out.data_ptr() or None,
               None if g_residual is None else (g_residual.data_ptr() or None), eps, weight_bias,
               g_h.data_ptr() or None, gw.data_ptr(), rows, D, code)
    if st:
        _native.check("rmsnorm_fused_vjp", st)
    return g_h, gw


class BoundCall:
    """One C call with its tensors checked once (rmsnorm_fwd_bind,
    rmsnorm_vjp_bind): calling it launches the kernels on the device's
    current stream (or the stream given at bind time).  For loops that run
    the same op on the same buffers every step (a decode loop's per-token
    norm): it keeps the tensors alive, and they must keep their storage,
    shape and dtype for as long as the bound call is used."""

    __slots__ = ("_fn", "_args", "_dev", "_stream", "_name", "_keep", "outputs")

    def __init__(self, name, fn, args, dev, stream, keep, outputs):
        self._name = name
        self._fn = fn
        self._args = args
        self._dev = dev
        self._stream = stream
        self._keep = keep
        self.outputs = outputs

    def __call__(self):
        st = _call(self._dev, self._stream, self._fn, *self._args)
        if st:
            _native.check(self._name, st)
        return self.outputs


def rmsnorm_fwd_bind(x: torch.Tensor, w: torch.Tensor, eps: float, weight_bias: float = 0.0,
                     residual: Optional[torch.Tensor] = None, *, out: Optional[torch.Tensor] = None,
                     new_residual: Optional[torch.Tensor] = None, stream=None) -> BoundCall:
    """rmsnorm_fwd with its arguments checked now and the call issued by the
    returned BoundCall (which returns (out, new_residual))."""
    rows, D, dev, code = _rows_dev(x)
    _weight(w, x, D, dev)
    if out is None:
        out = torch.empty_like(x)
    _like("out", out, x, dev)
    if residual is not None:
        _like("residual", residual, x, dev)
        if new_residual is None:
            new_residual = torch.empty_like(x)
        _like("new_residual", new_residual, x, dev)
    elif new_residual is not None:
        raise ValueError("new_residual given without residual")
    args = (x.data_ptr() or None, None if residual is None else (residual.data_ptr() or None),
            w.data_ptr(), eps, weight_bias, out.data_ptr() or None,
            None if new_residual is None else (new_residual.data_ptr() or None), rows, D, code)
    return BoundCall("rmsnorm_fwd", _fn("rmsnorm_fwd"), args, dev, stream,
                     (x, w, residual), (out, new_residual))


def rmsnorm_vjp_bind(x: torch.Tensor, w: torch.Tensor, g: torch.Tensor, eps: float,
                     weight_bias: float = 0.0, *, gx: Optional[torch.Tensor] = None,
                     gw: Optional[torch.Tensor] = None, stream=None) -> BoundCall:
    """rmsnorm_vjp with its arguments checked now and the call issued by the
    returned BoundCall (which returns (gx, gw))."""
    rows, D, dev, code = _rows_dev(x)
    _weight(w, x, D, dev)
    _like("g", g, x, dev)
    if gx is None:
        gx = torch.empty_like(x)
    _like("gx", gx, x, dev)
    gw = _gw(gw, D, dev)
    args = (x.data_ptr() or None, w.data_ptr(), g.data_ptr() or None, eps, weight_bias,
            gx.data_ptr() or None, gw.data_ptr(), rows, D, code)
    return BoundCall("rmsnorm_vjp", _fn("rmsnorm_vjp"), args, dev, stream, (x, w, g), (gx, gw))


def _vjp_outputs(x, g, gx, gw, D):
    _check_like("g", g, x)
    if gx is None:
        gx = torch.empty_like(x)
    _check_like("gx", gx, x)
    if gw is None:
        gw = torch.empty(D, dtype=torch.float32, device=x.device)
    if (gw.dtype != torch.float32 or gw.shape != (D,) or gw.device != x.device
            or not gw.is_contiguous()):
        raise ValueError("gw must be a contiguous [%d] float32 tensor on %s" % (D, x.device))
    return gx, gw


def rmsnorm_gated_silu(x: torch.Tensor, *, out: Optional[torch.Tensor] = None, stream=None):
    """silu(x[..., :d]) * x[..., d:] for x of last dimension 2d; returns the
    [..., d] result."""
    if x.shape[-1] % 2:
        raise ValueError("the last dimension of x must be even (2d)")
    rows, two_d = _rows_d(x)
    d = two_d // 2
    code = _dtype_code(x, (0, 1))
    if out is None:
        out = torch.empty(*x.shape[:-1], d, dtype=x.dtype, device=x.device)
    if (out.dtype != x.dtype or out.device != x.device or out.shape != (*x.shape[:-1], d)
            or not out.is_contiguous()):
        raise ValueError("out must be a contiguous %s tensor of shape %s" % (
            x.dtype, tuple((*x.shape[:-1], d))))
    with _OnDevice(x.device):
        st = _native.lib().rmsnorm_gated_silu(_ptr(x), _ptr(out), rows, d, code,
                                              _stream(x.device, stream))
    _native.check("rmsnorm_gated_silu", st)
    return out


def rmsnorm_rope_kv_append(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                           positions: torch.Tensor, slots: torch.Tensor, k_cache: torch.Tensor,
                           v_cache: torch.Tensor, *, rope_base: float = 10000.0,
                           cos_sin: Optional[torch.Tensor] = None, interleaved: bool = False,
                           q_out: Optional[torch.Tensor] = None, stream=None):
    """Rotates q (into q_out; pass q_out=q for in place) and k, and writes k and
    v into rows `slots` of the caches.  q: [T, Hq, Dh]; k, v: [T, Hkv, Dh];
    positions, slots: [T] int64 CUDA tensors; caches [num_slots, Hkv, Dh];
    cos_sin: optional [max_pos, Dh] float32 table.  Returns q_out."""
    if q.dim() != 3 or k.dim() != 3 or v.shape != k.shape:
        raise ValueError("q must be [T, Hq, Dh] and k, v [T, Hkv, Dh]")
    T, Hq, Dh = q.shape
    Hkv = k.shape[1]
    if k.shape[0] != T or k.shape[2] != Dh:
        raise ValueError("k and v must be [T, Hkv, Dh] with q's T and Dh")
    code = _dtype_code(q, (0, 1))
    for name, t in (("k", k), ("v", v), ("k_cache", k_cache), ("v_cache", v_cache)):
        if t.dtype != q.dtype or t.device != q.device or not t.is_contiguous():
            raise ValueError("%s must be a contiguous %s tensor on %s" % (name, q.dtype, q.device))
    if not q.is_cuda or not q.is_contiguous():
        raise ValueError("q must be a contiguous CUDA tensor")
    if k_cache.dim() != 3 or k_cache.shape[1:] != (Hkv, Dh) or v_cache.shape != k_cache.shape:
        raise ValueError("caches must be [num_slots, Hkv, Dh]")
    for name, t in (("positions", positions), ("slots", slots)):
        if t.dtype != torch.int64 or t.shape != (T,) or t.device != q.device or not t.is_contiguous():
            raise ValueError("%s must be a contiguous [T] int64 tensor on %s" % (name, q.device))
    max_pos = 0
    if cos_sin is not None:
        if (cos_sin.dtype != torch.float32 or cos_sin.dim() != 2 or cos_sin.shape[1] != Dh
                or cos_sin.device != q.device or not cos_sin.is_contiguous()):
            raise ValueError("cos_sin must be a contiguous [max_pos, Dh] float32 tensor")
        max_pos = cos_sin.shape[0]
    if q_out is None:
        q_out = torch.empty_like(q)
    _check_like("q_out", q_out, q)
    with _OnDevice(q.device):
        st = _native.lib().rmsnorm_rope_kv_append(
            _ptr(q), _ptr(k), _ptr(v), _ptr(positions), _ptr(slots), _ptr(q_out), _ptr(k_cache),
            _ptr(v_cache), _ptr(cos_sin), max_pos, rope_base, 1 if interleaved else 0, T, Hq, Hkv,
            Dh, k_cache.shape[0], code, _stream(q.device, stream))
    _native.check("rmsnorm_rope_kv_append", st)
    return q_out


def _check_rstd(rstd: torch.Tensor, rows: int, device: torch.device) -> None:
    if (rstd.dtype != torch.float32 or rstd.numel() != rows or rstd.device != device
            or not rstd.is_contiguous()):
        raise ValueError("rstd must be a contiguous float32 tensor of %d elements on %s" % (
            rows, device))


def rmsnorm_fwd_ex(x: torch.Tensor, w: torch.Tensor, eps: float, weight_bias: float = 0.0,
                   residual: Optional[torch.Tensor] = None, *, out: Optional[torch.Tensor] = None,
                   new_residual: Optional[torch.Tensor] = None, rstd=None, stream=None):
    """The forward on rows a stride apart (each of x, residual, out,
    new_residual may be a slice of a wider buffer), optionally writing the
    per-row scale.  rstd: None (not written), True (allocated here) or a
    [rows] float32 tensor.  Returns (out, new_residual, rstd); new outputs
    are allocated dense."""
    rows, D, ld_x = _rows_ld("x", x)
    code = _dtype_code(x)
    _check_w(w, x, D)
    ld_r = ld_n = D
    if residual is not None:
        ld_r = _check_rows_like("residual", residual, x)
        if new_residual is None:
            new_residual = torch.empty(x.shape, dtype=x.dtype, device=x.device)
        ld_n = _check_rows_like("new_residual", new_residual, x)
    elif new_residual is not None:
        raise ValueError("new_residual given without residual")
    if out is None:
        out = torch.empty(x.shape, dtype=x.dtype, device=x.device)
    ld_o = _check_rows_like("out", out, x)
    if rstd is True:
        rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    if rstd is not None:
        _check_rstd(rstd, rows, x.device)
    with _OnDevice(x.device):
        st = _native.lib().rmsnorm_fwd_ex(_ptr(x), ld_x, _ptr(residual), ld_r, _ptr(w), eps,
                                          weight_bias, _ptr(out), ld_o, _ptr(new_residual), ld_n,
                                          _ptr(rstd), rows, D, code, _stream(x.device, stream))
    _native.check("rmsnorm_fwd_ex", st)
    return out, new_residual, rstd


def rmsnorm_vjp_ex(x: torch.Tensor, w: torch.Tensor, g: torch.Tensor, eps: float,
                   weight_bias: float = 0.0, g_residual: Optional[torch.Tensor] = None, *,
                   rstd: Optional[torch.Tensor] = None, gx: Optional[torch.Tensor] = None,
                   gw: Optional[torch.Tensor] = None, stream=None):
    """The VJP (of the fused op when g_residual is given) on rows a stride
    apart, optionally with the forward's per-row scale rstd ([rows] float32)
    in place of recomputing it.  Returns (gx, gw)."""
    rows, D, ld_x = _rows_ld("x", x)
    code = _dtype_code(x)
    _check_w(w, x, D)
    ld_g = _check_rows_like("g", g, x)
    ld_gr = D
    if g_residual is not None:
        ld_gr = _check_rows_like("g_residual", g_residual, x)
    if gx is None:
        gx = torch.empty(x.shape, dtype=x.dtype, device=x.device)
    ld_gx = _check_rows_like("gx", gx, x)
    if gw is None:
        gw = torch.empty(D, dtype=torch.float32, device=x.device)
    if (gw.dtype != torch.float32 or gw.shape != (D,) or gw.device != x.device
            or not gw.is_contiguous()):
        raise ValueError("gw must be a contiguous [%d] float32 tensor on %s" % (D, x.device))
    if rstd is not None:
        _check_rstd(rstd, rows, x.device)
    with _OnDevice(x.device):
        st = _native.lib().rmsnorm_vjp_ex(_ptr(x), ld_x, _ptr(w), _ptr(g), ld_g, _ptr(g_residual),
                                          ld_gr, _ptr(rstd), eps, weight_bias, _ptr(gx), ld_gx,
                                          _ptr(gw), rows, D, code, _stream(x.device, stream))
    _native.check("rmsnorm_vjp_ex", st)
    return gx, gw


def rmsnorm_vjp_workspace_size(rows: int, D: int, dtype: torch.dtype) -> int:
    """Bytes of scratch rmsnorm_vjp_ws needs on the current device."""
    return int(_native.lib().rmsnorm_vjp_workspace_size(rows, D, _DTYPES[dtype]))


def rmsnorm_vjp_ws(x: torch.Tensor, w: torch.Tensor, g: torch.Tensor, eps: float,
                   weight_bias: float = 0.0, *, workspace: Optional[torch.Tensor] = None,
                   gx: Optional[torch.Tensor] = None, gw: Optional[torch.Tensor] = None,
                   stream=None):
    """rmsnorm_vjp with caller-owned scratch (a uint8 CUDA tensor of at least
    rmsnorm_vjp_workspace_size bytes; allocated here through torch when not
    given)."""
    rows, D = _rows_d(x)
    code = _dtype_code(x)
    _check_w(w, x, D)
    gx, gw = _vjp_outputs(x, g, gx, gw, D)
    with _OnDevice(x.device):
        if workspace is None:
            nbytes = rmsnorm_vjp_workspace_size(rows, D, x.dtype)
            workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=x.device)
        if workspace.device != x.device or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous tensor on %s" % x.device)
        nbytes = workspace.numel() * workspace.element_size()
        st = _native.lib().rmsnorm_vjp_ws(_ptr(x), _ptr(w), _ptr(g), eps, weight_bias,
                                          _ptr(gx), _ptr(gw), rows, D, code, _ptr(workspace),
                                          nbytes, _stream(x.device, stream))
    _native.check("rmsnorm_vjp_ws", st)
    return gx, gw


def rmsnorm_vjp_noalloc(x: torch.Tensor, w: torch.Tensor, g: torch.Tensor, eps: float,
                        weight_bias: float = 0.0, *, gx: Optional[torch.Tensor] = None,
                        gw: Optional[torch.Tensor] = None, stream=None):
    """rmsnorm_vjp with its gw partial rows in the library's fixed device array
    (nothing allocated by the library; gx and gw are allocated here through
    torch when not given).  Problems whose partials do not fit the array raise
    with RMSNORM_ERR_UNSUPPORTED."""
    rows, D = _rows_d(x)
    code = _dtype_code(x)
    _check_w(w, x, D)
    gx, gw = _vjp_outputs(x, g, gx, gw, D)
    with _OnDevice(x.device):
        st = _native.lib().rmsnorm_vjp_noalloc(_ptr(x), _ptr(w), _ptr(g), eps, weight_bias,
                                               _ptr(gx), _ptr(gw), rows, D, code,
                                               _stream(x.device, stream))
    _native.check("rmsnorm_vjp_noalloc", st)
    return gx, gw


def rmsnorm_device_status(clear: bool = True) -> int:
    """Device status bits of the current device (synchronises).  The bits are
    returned, not raised: the status the C call derives from them (timeout,
    bad index) is not an error of the call itself."""
    bits = ctypes.c_uint(0)
    st = _native.lib().rmsnorm_device_status(ctypes.byref(bits), 1 if clear else 0)
    if st != 0 and not (bits.value and st in (1, 5)):
        _native.check("rmsnorm_device_status", st)
    return int(bits.value)


def rmsnorm_debug_inject(drop_tile: int = -1, budget_cycles: int = 0) -> None:
    """Test hook: drop one staged tile's copy and shorten the wait budget
    ((-1, 0) restores normal operation)."""
    _native.check("rmsnorm_debug_inject",
                  _native.lib().rmsnorm_debug_inject(drop_tile, budget_cycles))


def rmsnorm_debug_claim_counters(count: int) -> None:
    """Test hook: staged forwards launched outside a capture cycle through the
    first `count` claim-counter sets (1 makes consecutive forwards share one;
    0 restores the default)."""
    _native.check("rmsnorm_debug_claim_counters",
                  _native.lib().rmsnorm_debug_claim_counters(count))


def rmsnorm_debug_fail_allocs(count: int) -> None:
    """Test hook: the next `count` gw scratch allocations of the pooled VJP
    entry points report RMSNORM_ERR_NO_MEMORY without allocating (0 cancels)."""
    _native.check("rmsnorm_debug_fail_allocs", _native.lib().rmsnorm_debug_fail_allocs(count))


def rmsnorm_describe_dispatch(op: str, rows: int, D: int, dtype: torch.dtype,
                              has_residual: bool = False, aligned: bool = True) -> str:
    """The kernel plan the library would choose ('fwd' or 'vjp').  aligned:
    True/1 dense 16-byte aligned tensors, 2 dense tensors at one shared
    unaligned offset, False/0 anything else."""
    s = _native.lib().rmsnorm_describe_dispatch(1 if op == "vjp" else 0, rows, D, _DTYPES[dtype],
                                                1 if has_residual else 0, int(aligned))
    return s.decode()


def rmsnorm_status_string(status: int) -> str:
    return _native.lib().rmsnorm_status_string(status).decode()
