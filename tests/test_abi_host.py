"""Host-side checks of the C ABI (no GPU needed, no kernel launched).

The library must load on a machine without a GPU, export every symbol
include/addln.h declares, and reject bad arguments before its first CUDA
call.  Pointers below are fake addresses: every call here fails validation,
so none is ever dereferenced.
"""
from __future__ import annotations

import os
import re
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "addln.h")


@pytest.fixture(scope="module")
def lib():
    from memory_bound_add_gb300.build import build
    build()
    from memory_bound_add_gb300 import binding
    return binding.lib()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def header_defines():
    vals = {}
    for m in re.finditer(r"#define\s+(ADDLN_\w+)\s+\(?(-?\d+)\)?", open(HEADER).read()):
        vals[m.group(1)] = int(m.group(2))
    return vals


def test_header_declares_the_expected_entry_points():
    assert header_functions() == sorted([
        "add_layernorm_fwd", "add_layernorm_fwd_host", "add_layernorm_fwd_host_workspace_size",
        "add_layernorm_fwd_host_last_mode",
        "add_fwd", "layernorm_fwd", "softmax_fwd", "bias_gelu_residual_fwd",
        "bias_add_fwd", "gelu_fwd", "add_layernorm_bwd", "add_layernorm_bwd_workspace_size",
        "add_layernorm_bwd_noalloc",
        "addln_strerror",
        "addln_max_hidden", "addln_bounds_checked", "addln_bounds_violation",
        "addln_get_device_error", "addln_set_force_path", "addln_set_wait_limit_ns",
        "addln_set_grid_cap", "addln_set_pdl", "addln_set_cta_shape", "addln_set_warp_rows",
        "addln_last_path",
        "addln_last_cuda_error"])


def test_library_exports_every_header_symbol(lib):
    from memory_bound_add_gb300.build import LIB
    out = subprocess.run(["nm", "-D", "--defined-only", LIB], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in header_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_binding_signatures_cover_the_header():
    from memory_bound_add_gb300 import binding
    assert sorted(binding.SIGNATURES) == header_functions()
    d = header_defines()
    assert (binding.FP32, binding.FP16, binding.BF16) == (d["ADDLN_FP32"], d["ADDLN_FP16"],
                                                          d["ADDLN_BF16"])
    for k in ("NULL", "SHAPE", "DTYPE", "EPS", "ALIAS", "LAUNCH", "UNSUPPORTED",
              "DEVICE_TIMEOUT", "CUDA", "WORKSPACE", "BOUNDS"):
        assert getattr(binding, "ERR_" + k) == d["ADDLN_ERR_" + k]
    for k in ("AUTO", "WARP_VEC", "CTA_TMA", "CTA_VEC", "SCALAR"):
        assert getattr(binding, "PATH_" + k) == d["ADDLN_PATH_" + k]
    for k in ("PIPELINED", "MAPPED"):
        assert getattr(binding, "HOST_" + k) == d["ADDLN_HOST_" + k]


def test_strerror_and_limits(lib):
    from memory_bound_add_gb300 import binding as b
    for code in range(-10, 1):
        assert lib.addln_strerror(code)
    assert b"unknown" in lib.addln_strerror(-99)
    assert lib.addln_max_hidden(b.FP32) == 16384
    assert lib.addln_max_hidden(b.FP16) == 32768
    assert lib.addln_max_hidden(b.BF16) == 32768
    assert lib.addln_max_hidden(7) == b.ERR_DTYPE
    assert lib.addln_last_path() == b"none"
    assert lib.addln_last_cuda_error() == b"none"


def test_force_path_setter(lib):
    from memory_bound_add_gb300 import binding as b
    assert lib.addln_set_force_path(b.PATH_SCALAR) == b.PATH_AUTO
    assert lib.addln_set_force_path(b.PATH_AUTO) == b.PATH_SCALAR
    assert lib.addln_set_force_path(99) == b.ERR_SHAPE
    assert lib.addln_set_wait_limit_ns(5) == 1000000000
    assert lib.addln_set_wait_limit_ns(1000000000) == 5
    assert lib.addln_set_grid_cap(3) == 0
    assert lib.addln_set_grid_cap(0) == 3
    assert lib.addln_set_pdl(0) == 1
    assert lib.addln_set_pdl(1) == 0
    assert lib.addln_set_cta_shape(256, 3) == 0
    assert lib.addln_set_cta_shape(0, 0) == 256
    assert lib.addln_set_cta_shape(100, 0) == b.ERR_SHAPE
    assert lib.addln_set_cta_shape(0, 9) == b.ERR_SHAPE


BASE = 0x7F0000000000   # fake, 16-byte aligned


def fused(lib, x=BASE, r=BASE + 0x1000000, g=BASE + 0x2000000, bt=BASE + 0x2100000,
          y=BASE + 0x3000000, a=None, mean=None, rstd=None, rows=4, H=8, eps=1e-5, dtype=0):
    return lib.add_layernorm_fwd(x, r, g, bt, y, a, mean, rstd, rows, H, eps, dtype, None)


def test_validation_codes(lib):
    from memory_bound_add_gb300 import binding as b
    assert fused(lib, dtype=3) == b.ERR_DTYPE
    assert fused(lib, dtype=-1) == b.ERR_DTYPE
    assert fused(lib, H=0) == b.ERR_SHAPE
    assert fused(lib, H=-5) == b.ERR_SHAPE
    assert fused(lib, rows=-1) == b.ERR_SHAPE
    assert fused(lib, H=16385, dtype=b.FP32) == b.ERR_SHAPE
    assert fused(lib, H=32769, dtype=b.BF16) == b.ERR_SHAPE
    assert fused(lib, rows=(1 << 62), H=8) == b.ERR_SHAPE
    assert fused(lib, eps=-1e-6) == b.ERR_EPS
    assert fused(lib, eps=float("nan")) == b.ERR_EPS
    assert fused(lib, eps=float("inf")) == b.ERR_EPS
    assert fused(lib, x=None) == b.ERR_NULL
    assert fused(lib, r=None) == b.ERR_NULL
    assert fused(lib, g=None) == b.ERR_NULL
    assert fused(lib, bt=None) == b.ERR_NULL
    assert fused(lib, y=None) == b.ERR_NULL
    # rows == 0 is a no-op once dtype, H and eps are valid, even with NULLs
    assert fused(lib, rows=0, x=None, y=None) == b.OK
    assert fused(lib, rows=0, dtype=9) == b.ERR_DTYPE


def host_fused(lib, x=BASE, r=BASE + 0x1000000, g=BASE + 0x2000000, bt=BASE + 0x2100000,
               y=BASE + 0x3000000, a=None, mean=None, rstd=None, rows=4, H=8, eps=1e-5, dtype=0,
               ws=BASE + 0x4000000, ws_bytes=1 << 20):
    return lib.add_layernorm_fwd_host(x, r, g, bt, y, a, mean, rstd, rows, H, eps, dtype, ws,
                                      ws_bytes, None)


def test_host_entry_validation_before_any_cuda_call(lib):
    # every rejection below is decided on the host, before the first CUDA call
    from memory_bound_add_gb300 import binding as b
    mode0 = lib.add_layernorm_fwd_host_last_mode()
    assert host_fused(lib, dtype=3) == b.ERR_DTYPE
    assert host_fused(lib, H=0) == b.ERR_SHAPE
    assert host_fused(lib, rows=-1) == b.ERR_SHAPE
    assert host_fused(lib, eps=-1.0) == b.ERR_EPS
    assert host_fused(lib, eps=float("nan")) == b.ERR_EPS
    for k in ("x", "r", "g", "bt", "y"):
        assert host_fused(lib, **{k: None}) == b.ERR_NULL
    assert host_fused(lib, rows=0, x=None, y=None) == b.OK
    need = lib.add_layernorm_fwd_host_workspace_size(4, 8, b.FP32, 0, 0)
    assert need > 0
    assert host_fused(lib, ws=None) == b.ERR_WORKSPACE
    assert host_fused(lib, ws_bytes=need - 1) == b.ERR_WORKSPACE
    assert host_fused(lib, ws=BASE + 0x4000010, ws_bytes=need) == b.ERR_WORKSPACE  # not 256-aligned
    # y may be x exactly, not partly; a must lie apart from y
    assert host_fused(lib, y=BASE + 64, ws_bytes=need) == b.ERR_ALIAS
    assert host_fused(lib, a=BASE + 0x3000000, ws_bytes=need) == b.ERR_ALIAS
    assert host_fused(lib, mean=BASE + 0x2000000 + 8, rstd=BASE + 0x5000000, ws_bytes=need) == b.ERR_ALIAS
    # workspace sizes: outputs add buffers; chunks of about 4 MiB of X
    assert lib.add_layernorm_fwd_host_workspace_size(0, 8, b.FP32, 0, 0) == 0
    assert lib.add_layernorm_fwd_host_workspace_size(4, 8, 7, 0, 0) == b.ERR_DTYPE
    base = lib.add_layernorm_fwd_host_workspace_size(2048, 4096, b.FP16, 0, 0)
    assert lib.add_layernorm_fwd_host_workspace_size(2048, 4096, b.FP16, 1, 0) > base
    assert lib.add_layernorm_fwd_host_workspace_size(2048, 4096, b.FP16, 0, 1) > base
    # two 512-row chunk buffers of X, R, Y (4 MiB each) plus gamma and beta
    assert base == 2 * 3 * 512 * 4096 * 2 + 2 * 4096 * 4
    # rejected calls (and rows == 0) record no mode: none queued any work
    assert lib.add_layernorm_fwd_host_last_mode() == mode0


def test_valid_host_call_without_a_gpu_fails_cleanly(lib):
    # past every host-side check, the first CUDA call (the device query that
    # picks the transfer mode) reports the missing GPU as an error code;
    # no pointer is touched before it
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: the call would run on the placeholder pointers")
    from memory_bound_add_gb300 import binding as b
    assert host_fused(lib) == b.ERR_CUDA


def bwd_call(lib, fn, dy=BASE, a=BASE + 0x1000000, mean=BASE + 0x2000000,
             rstd=BASE + 0x2100000, gamma=BASE + 0x2200000, dres=None, dx=BASE + 0x3000000,
             dg=BASE + 0x4000000, db=BASE + 0x4100000, rows=4, H=8, dtype=0):
    args = (dy, a, mean, rstd, gamma, dres, dx, dg, db, rows, H, dtype)
    if fn == "add_layernorm_bwd":
        return lib.add_layernorm_bwd(*args, BASE + 0x5000000, 1 << 20, None)
    return lib.add_layernorm_bwd_noalloc(*args, None)


@pytest.mark.parametrize("kw", [
    {"dtype": 3}, {"dtype": -1}, {"H": 0}, {"H": -2}, {"rows": -1}, {"H": 16385},
    {"H": 32769, "dtype": 2}, {"rows": 1 << 62},
    {"dg": None},                    # dgamma without dbeta
    {"db": None},                    # dbeta without dgamma
    {"rows": 0, "dg": None},         # the pair rule holds for an empty batch too
    {"rows": 0, "dg": None, "db": None, "dy": None},     # an empty batch is a no-op
])
def test_noalloc_backward_returns_the_workspace_entry_points_codes(lib, kw):
    # the no-alloc entry point checks its arguments as add_layernorm_bwd does,
    # in the same order, before any CUDA call
    a = bwd_call(lib, "add_layernorm_bwd", **kw)
    b = bwd_call(lib, "add_layernorm_bwd_noalloc", **kw)
    assert a == b, kw
    assert a <= 0


def test_noalloc_backward_null_inputs(lib):
    from memory_bound_add_gb300 import binding as b
    # no column sums: add_layernorm_bwd's own NULL checks decide
    for k in ("dy", "a", "mean", "rstd", "gamma", "dx"):
        assert bwd_call(lib, "add_layernorm_bwd_noalloc", dg=None, db=None, **{k: None}) == b.ERR_NULL
        assert bwd_call(lib, "add_layernorm_bwd_noalloc", **{k: None}) == b.ERR_NULL


def test_alias_rules(lib):
    from memory_bound_add_gb300 import binding as b
    rows, H = 4, 8
    tb = rows * H * 4
    x = BASE
    # partial overlaps of an output with an input
    assert fused(lib, x=x, y=x + 16) == b.ERR_ALIAS
    assert fused(lib, x=x, y=x - 16) == b.ERR_ALIAS
    assert fused(lib, r=x + 0x1000000, a=x + 0x1000000 + 32, y=x + 0x3000000) == b.ERR_ALIAS
    # output over gamma or beta, even exactly
    assert fused(lib, y=BASE + 0x2000000) == b.ERR_ALIAS
    assert fused(lib, mean=BASE + 0x2100000 + 4, rstd=BASE + 0x5000000) == b.ERR_ALIAS
    # outputs against each other
    y = BASE + 0x3000000
    assert fused(lib, y=y, a=y) == b.ERR_ALIAS
    assert fused(lib, y=y, a=y + tb - 16) == b.ERR_ALIAS
    m = BASE + 0x6000000
    assert fused(lib, mean=m, rstd=m + 8) == b.ERR_ALIAS
    assert fused(lib, mean=m, rstd=y + 64) == b.ERR_ALIAS
    # the unfused kernels
    assert lib.add_fwd(x, x + 0x1000000, x + 8, 64, 0, None) == b.ERR_ALIAS
    assert lib.add_fwd(x, None, x + 0x4000000, 64, 0, None) == b.ERR_NULL
    assert lib.add_fwd(x, x, x, -1, 0, None) == b.ERR_SHAPE
    assert lib.add_fwd(x, x, x, 64, 5, None) == b.ERR_DTYPE
    assert lib.add_fwd(None, None, None, 0, 0, None) == b.OK
    assert lib.layernorm_fwd(x, BASE + 0x2000000, BASE + 0x2100000, x + 4, None, None, rows, H,
                             1e-5, 0, None) == b.ERR_ALIAS
    assert lib.layernorm_fwd(x, None, BASE + 0x2100000, y, None, None, rows, H, 1e-5, 0,
                             None) == b.ERR_NULL
    # softmax
    assert lib.softmax_fwd(x, x + 4, rows, H, 0, None) == b.ERR_ALIAS
    assert lib.softmax_fwd(None, y, rows, H, 0, None) == b.ERR_NULL
    assert lib.softmax_fwd(x, y, rows, 0, 0, None) == b.ERR_SHAPE
    assert lib.softmax_fwd(x, y, rows, H, 4, None) == b.ERR_DTYPE
    assert lib.softmax_fwd(x, y, rows, 32769, 1, None) == b.ERR_SHAPE
    assert lib.softmax_fwd(None, None, 0, H, 0, None) == b.OK
    # bias + GELU + residual and its chain
    bias = BASE + 0x2000000
    assert lib.bias_gelu_residual_fwd(x, x + 0x1000000, bias, x + 8, rows, H, 0, None) == b.ERR_ALIAS
    assert lib.bias_gelu_residual_fwd(x, x + 0x1000000, bias, bias, rows, H, 0, None) == b.ERR_ALIAS
    assert lib.bias_gelu_residual_fwd(x, None, bias, y, rows, H, 0, None) == b.ERR_NULL
    assert lib.bias_gelu_residual_fwd(x, x, bias, y, rows, 0, 0, None) == b.ERR_SHAPE
    assert lib.bias_gelu_residual_fwd(x, x, bias, y, rows, H, 7, None) == b.ERR_DTYPE
    assert lib.bias_gelu_residual_fwd(None, None, None, None, 0, H, 0, None) == b.OK
    assert lib.bias_add_fwd(x, None, y, rows, H, 0, None) == b.ERR_NULL
    assert lib.bias_add_fwd(x, bias, x + 4, rows, H, 0, None) == b.ERR_ALIAS
    assert lib.gelu_fwd(x, x + 4, 64, 0, None) == b.ERR_ALIAS
    assert lib.gelu_fwd(x, y, -1, 0, None) == b.ERR_SHAPE
    # backward (fake pointers: every call fails its checks before CUDA)
    dy, a, mu, rs, g = x, BASE + 0x1000000, BASE + 0x4000000, BASE + 0x4100000, BASE + 0x2000000
    dx, dg, db, ws = BASE + 0x5000000, BASE + 0x6000000, BASE + 0x6100000, BASE + 0x7000000

    def bwd(**kw):
        args = dict(dy=dy, a=a, mu=mu, rs=rs, g=g, dres=None, dx=dx, dg=dg, db=db, rows=rows, H=H,
                    dtype=0, ws=ws, wsb=1 << 20)
        args.update(kw)
        return lib.add_layernorm_bwd(args["dy"], args["a"], args["mu"], args["rs"], args["g"],
                                     args["dres"], args["dx"], args["dg"], args["db"],
                                     args["rows"], args["H"], args["dtype"], args["ws"],
                                     args["wsb"], None)
    assert bwd(dtype=5) == b.ERR_DTYPE
    assert bwd(H=0) == b.ERR_SHAPE
    assert bwd(db=None) == b.ERR_NULL                 # dgamma without dbeta
    assert bwd(a=None) == b.ERR_NULL
    assert bwd(wsb=-1) == b.ERR_WORKSPACE
    assert bwd(dx=dy + 4) == b.ERR_ALIAS              # partial overlap with dY
    assert bwd(dg=g) == b.ERR_ALIAS                   # dgamma over gamma
    assert bwd(ws=dx) == b.ERR_ALIAS                  # workspace over dX
    assert bwd(db=dg + 4) == b.ERR_ALIAS
    assert lib.add_layernorm_bwd_workspace_size(4, 8, 9) == b.ERR_DTYPE
    assert lib.add_layernorm_bwd_workspace_size(4, 0, 0) == b.ERR_SHAPE
    assert lib.add_layernorm_bwd_workspace_size(0, 8, 0) == 0


def test_missing_library_fails_loudly(tmp_path):
    code = (
        "import sys; sys.path.insert(0, %r)\n"
        "from memory_bound_add_gb300 import binding\n"
        "binding.LIB_PATH = %r\n"
        "try:\n"
        "    binding.lib()\n"
        "except RuntimeError as e:\n"
        "    print('raised', e)\n"
        "else:\n"
        "    print('loaded')\n" % (ROOT, str(tmp_path / "nope.so")))
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, check=True)
    assert out.stdout.startswith("raised")


def test_product_path_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "memory_bound_add_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle", text, flags=re.M), f
                assert "liboracle" not in text and "addln_oracle" not in text, f
    for f in ("addln.h",):
        assert "oracle" not in open(os.path.join(ROOT, "include", f)).read()


def test_oracle_shares_no_code_with_the_library():
    src = open(os.path.join(ROOT, "oracle", "addln_oracle.c")).read()
    assert "#include \"" not in src          # only system headers
    for dirpath, _, files in os.walk(os.path.join(ROOT, "oracle")):
        for f in files:
            if f.endswith(".py"):
                text = open(os.path.join(dirpath, f)).read()
                assert "memory_bound_add_gb300" not in text, f


def test_tolerance_helper_ulp():
    sys.path.insert(0, os.path.dirname(__file__))
    from _parity import ulp, y_violations
    assert ulp(np.array([1.0]), "bf16")[0] == 2.0 ** -7
    assert ulp(np.array([10.0]), "bf16")[0] == 2.0 ** -4
    assert ulp(np.array([1.0]), "fp16")[0] == 2.0 ** -10
    assert ulp(np.array([0.0]), "fp16")[0] == 2.0 ** -24
    ref = np.array([10.03])
    assert not y_violations(np.array([10.0625]), ref, "bf16").any()   # one rounding step away
    assert y_violations(np.array([10.25]), ref, "bf16").any()
    assert y_violations(np.array([1.0 + 5e-3]), np.array([1.0]), "fp16").any()
    assert not y_violations(np.array([1.0 + 1e-5]), np.array([1.0]), "fp32").any()
    assert y_violations(np.array([1.0 + 3e-5]), np.array([1.0]), "fp32").any()


def test_bounds_checked_build_loads_and_says_so():
    # the debugging build compiles every kernel with the bounds tests in, and
    # loads and answers on a machine without a GPU like the normal build
    from memory_bound_add_gb300 import binding
    from memory_bound_add_gb300.build import CHECKED_LIB, build
    path = build(checked=True)
    assert path == CHECKED_LIB
    checked = binding.load(CHECKED_LIB)
    assert checked.addln_bounds_checked() == 1
    assert binding.lib().addln_bounds_checked() == 0
    assert checked.addln_bounds_violation() == 0
    assert checked.addln_strerror(binding.ERR_BOUNDS).decode().startswith("a kernel skipped")
