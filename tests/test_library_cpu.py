"""The C-ABI library without a GPU: it builds, loads, exports every function
include/rmsnorm.h declares, and its host-side validation answers with status
codes before any CUDA call."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rmsnorm.h")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and
                                not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not available")


@pytest.fixture(scope="module")
def lib():
    from rmsnorm_fwd_bwd_add_gb300 import _native, build
    build.build()
    return _native.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rmsnorm_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    assert "rmsnorm_fwd" in names and "rmsnorm_vjp" in names
    from rmsnorm_fwd_bwd_add_gb300 import _native
    assert sorted(_native.EXPORTS) == names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert lib.rmsnorm_status_string(0) == b"ok"
    assert lib.rmsnorm_status_string(1) == b"invalid argument"
    assert lib.rmsnorm_status_string(5) == b"device-side wait timed out"
    assert lib.rmsnorm_status_string(99) == b"unknown status"


def _fwd(lib, x=1, res=None, w=1, eps=1e-6, wb=0.0, out=1, nr=None, rows=4, D=64, dtype=1):
    return lib.rmsnorm_fwd(x, res, w, eps, wb, out, nr, rows, D, dtype, None)


def test_host_validation_without_gpu(lib):
    # every case below is rejected before the library touches CUDA
    assert _fwd(lib, dtype=3) == 1
    assert _fwd(lib, D=0) == 1
    assert _fwd(lib, rows=-1) == 1
    assert _fwd(lib, eps=-1e-6) == 1
    assert _fwd(lib, eps=float("nan")) == 1
    assert _fwd(lib, eps=float("inf")) == 1
    assert _fwd(lib, wb=float("nan")) == 1
    assert _fwd(lib, w=None) == 1
    assert _fwd(lib, D=(1 << 24) + 1) == 2
    assert _fwd(lib, rows=1 << 62, D=1 << 20) == 2
    assert _fwd(lib, rows=0) == 0          # empty: nothing to do
    assert _fwd(lib, x=None) == 1
    assert _fwd(lib, out=None) == 1
    assert _fwd(lib, res=4096, nr=None) == 1   # residual without new_residual
    assert _fwd(lib, res=None, nr=4096) == 1
    # overlapping outputs / partial overlap with an input
    n = 4 * 64 * 2
    assert _fwd(lib, x=1 << 20, out=(1 << 20) + 16) == 1
    assert _fwd(lib, x=1 << 20, res=1 << 22, out=1 << 24, nr=(1 << 24) + n - 2) == 1
    vjp = lib.rmsnorm_vjp
    assert vjp(1, 1, 1, 1e-6, 0.0, 1, None, 4, 64, 0, None) == 1      # gw missing
    assert vjp(1, 1, 1, -1.0, 0.0, 1, 1, 4, 64, 0, None) == 1
    assert vjp(1 << 20, 1, 1 << 22, 1e-6, 0.0, (1 << 20) + 64, 1 << 24, 4, 64, 0, None) == 1
    ws = lib.rmsnorm_vjp_ws
    assert ws(1, 1, 1, 1e-6, 0.0, 1, None, 4, 64, 0, 1, 1 << 20, None) == 1
    assert lib.rmsnorm_vjp_workspace_size(4, 0, 0) == 0
    assert lib.rmsnorm_describe_dispatch(2, 4, 64, 0, 0, 1) == b"invalid"
    assert lib.rmsnorm_debug_inject(-1, 0) == 0


def _fwd_ex(lib, x, ld_x, out, ld_out, res=None, ld_res=0, nr=None, ld_nr=0, rstd=None, w=1 << 40,
            rows=8, D=64, dtype=1):
    return lib.rmsnorm_fwd_ex(x, ld_x, res, ld_res, w, 1e-6, 0.0, out, ld_out, nr, ld_nr, rstd,
                              rows, D, dtype, None)


def test_strided_validation_without_gpu(lib):
    """Row strides and rstd: rejections come before any CUDA call; layouts
    that pass it reach the device query, which fails here without a GPU
    (status 3), so they are only checked where no GPU is present."""
    import torch
    B, D, rows = 1 << 30, 64, 8
    row = 2 * D * 2  # bytes of one row of a [rows, 2D] bf16 buffer
    assert _fwd_ex(lib, B, D - 1, 1 << 32, D) == 1                       # row stride < D
    assert _fwd_ex(lib, B, 2 * D, B + 16, 2 * D) == 1                     # shifted by 16 bytes
    assert _fwd_ex(lib, B, 2 * D, B + D * 2 - 2, 2 * D) == 1              # last element shared
    assert _fwd_ex(lib, B, 2 * D, B + D * 2, 3 * D) == 1                  # other stride, extents meet
    assert _fwd_ex(lib, B, 2 * D, 1 << 32, D, rstd=B + row) == 1          # rstd inside x's span
    assert _fwd_ex(lib, B, 2 * D, 1 << 32, D, rstd=(1 << 40) + 8) == 1    # rstd over w
    assert _fwd_ex(lib, B, 2 * D, 1 << 32, D, res=B + D * 2, ld_res=2 * D,
                   nr=B + 8, ld_nr=2 * D) == 1                             # new_residual over x
    assert _fwd_ex(lib, B, 2 * D, 1 << 32, D, res=1 << 34, ld_res=D, nr=None) == 1
    vjp = lib.rmsnorm_vjp_ex
    gx = 1 << 32
    # g_residual partly over gx; rstd over gx; rstd over gw
    assert vjp(B, D, 1 << 40, 1 << 36, D, gx + 64, D, None, 1e-6, 0.0, gx, D, 1 << 38, rows, D, 1,
               None) == 1
    assert vjp(B, D, 1 << 40, 1 << 36, D, None, 0, gx + 32, 1e-6, 0.0, gx, D, 1 << 38, rows, D, 1,
               None) == 1
    assert vjp(B, D, 1 << 40, 1 << 36, D, None, 0, (1 << 38) + 4, 1e-6, 0.0, gx, D, 1 << 38, rows,
               D, 1, None) == 1
    assert vjp(B, D - 8, 1 << 40, 1 << 36, D, None, 0, None, 1e-6, 0.0, gx, D, 1 << 38, rows, D, 1,
               None) == 1
    if torch.cuda.is_available():
        return  # the accepted layouts below would launch on made-up addresses
    assert _fwd_ex(lib, B, 2 * D, B + D * 2, 2 * D) == 3                  # the other half: disjoint
    assert _fwd_ex(lib, B + D * 2, 2 * D, B, 2 * D) == 3                  # and the other way round
    assert _fwd_ex(lib, B, 2 * D, B, 2 * D) == 3                          # in place
    assert _fwd_ex(lib, B, D, B, 5 * D, rows=1) == 3                      # one row: no stride
    assert _fwd_ex(lib, B, 2 * D, 1 << 32, D, dtype=2) == 3               # fp32


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    from rmsnorm_fwd_bwd_add_gb300 import _native
    monkeypatch.setattr(_native, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(_native, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        _native.lib()


def test_no_cpu_tensors():
    import torch
    import rmsnorm_fwd_bwd_add_gb300 as rn
    x = torch.zeros(2, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        rn.rmsnorm_fwd(x, torch.ones(8, dtype=torch.bfloat16), 1e-6)


def test_product_does_not_import_oracle():
    pkg = os.path.join(ROOT, "rmsnorm_fwd_bwd_add_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b|rmsnorm_oracle", src, re.M), f


def test_alloc_failure_hook_arguments(lib):
    # the hook only sets a host-side counter: no GPU needed
    assert lib.rmsnorm_debug_fail_allocs(-1) == 1
    assert lib.rmsnorm_debug_fail_allocs(2) == 0
    assert lib.rmsnorm_debug_fail_allocs(0) == 0
