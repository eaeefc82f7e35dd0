"""The bounds-checked debugging build (ADDLN_CHECK_BOUNDS) on a small set of
shapes: every kernel family, every forced path, ragged rows, misaligned
buffers and capped persistent grids, through the checked library's own C ABI.

In that build each global load, store, bulk copy and L2 prefetch is first
tested against its buffer's extent; an access that would leave its buffer is
skipped and reported as ADDLN_ERR_BOUNDS.  Every call here must report none,
and every output must agree with the normal library's: the tests change no
arithmetic, but the two builds may contract a multiply and an add
differently, and the backward's grid (hence how its column partials are
grouped) follows each build's occupancy, so values agree to a couple of fp32
roundings (outputs an access skipped would be far off: zeros or stale
memory)."""
from __future__ import annotations

import ctypes

import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
mba = pytest.importorskip("memory_bound_add_gb300")
TD = synth.TORCH_DTYPES


@pytest.fixture(scope="module")
def chk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from memory_bound_add_gb300.build import CHECKED_LIB, build
    build()
    build(checked=True)
    lib = mba.binding.load(CHECKED_LIB)
    assert lib.addln_bounds_checked() == 1
    yield lib
    lib.addln_set_force_path(0)
    lib.addln_set_grid_cap(0)


def P(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def S():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def no_violation(lib, what):
    rc = lib.addln_get_device_error(S())
    assert rc == 0, f"{what}: {lib.addln_strerror(rc).decode()} (word {lib.addln_bounds_violation():#x})"


def assert_close(u, v, what):
    """Within two units in the last place of the output dtype (fp32: 2^-22
    relative) of the larger magnitude, plus 1e-6 absolute."""
    a, b = u.double(), v.double()
    rel = {torch.float32: 2.0 ** -22, torch.float16: 2.0 ** -10, torch.bfloat16: 2.0 ** -7}[u.dtype]
    bound = rel * torch.maximum(a.abs(), b.abs()) + 1e-6
    bad = ~((a - b).abs() <= bound)
    assert not bad.any(), f"{what}: {int(bad.sum())} values differ, e.g. {a[bad][:3]} vs {b[bad][:3]}"


def misaligned_copy(t):
    """t's values in a buffer that starts two bytes past a 16-byte boundary."""
    n = t.numel()
    buf = torch.empty(n + 16, dtype=t.dtype, device="cuda")
    v = buf[1:1 + n].view(t.shape)
    v.copy_(t)
    return v


FWD_CASES = [(rows, H, dt) for dt in ("fp32", "fp16", "bf16")
             for rows, H in ((37, 8), (37, 1000), (21, 1001), (13, 4096), (7, 4104), (3, 12288))]


@pytest.mark.parametrize("rows,H,dtype", FWD_CASES)
@pytest.mark.parametrize("path", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("cap", [0, 5])
def test_forward(chk, rows, H, dtype, path, cap):
    w = synth.custom(rows, H, dtype, want_resid=True, want_stats=True)
    d = synth.make_inputs(w, seed=H + rows)
    x, r = d["x"].cuda(), d["r"].cuda()
    g, b = d["gamma"].cuda(), d["beta"].cuda()
    code = mba.binding.DTYPE_CODE[TD[dtype]]
    outs = {}
    for lib, tag in ((mba.lib(), "normal"), (chk, "checked")):
        y, a = torch.empty_like(x), torch.empty_like(x)
        m = torch.empty(rows, device="cuda")
        s = torch.empty(rows, device="cuda")
        lib.addln_set_force_path(path)
        lib.addln_set_grid_cap(cap)
        rc = lib.add_layernorm_fwd(P(x), P(r), P(g), P(b), P(y), P(a), P(m), P(s), rows, H,
                                   1e-5, code, S())
        lib.addln_set_force_path(0)
        lib.addln_set_grid_cap(0)
        if rc == mba.binding.ERR_UNSUPPORTED:
            pytest.skip("the forced path cannot run this layout")
        assert rc == 0, lib.addln_strerror(rc).decode()
        torch.cuda.synchronize()
        if tag == "checked":
            no_violation(lib, f"forward {rows}x{H} {dtype} path {path} cap {cap}")
        outs[tag] = (y, a, m, s)
    for u, v in zip(outs["normal"], outs["checked"]):
        assert_close(u, v, f"forward {rows}x{H} {dtype} path {path}")


@pytest.mark.parametrize("dtype", ["fp16", "bf16", "fp32"])
@pytest.mark.parametrize("H", [8, 1000, 1001, 4096, 32000 // 4])
@pytest.mark.parametrize("path", [0, 1, 2, 4])
def test_softmax(chk, dtype, H, path):
    rows = 19
    x = (torch.randn(rows, H, generator=torch.Generator().manual_seed(H)) * 3).to(TD[dtype]).cuda()
    code = mba.binding.DTYPE_CODE[TD[dtype]]
    ys = []
    for lib in (mba.lib(), chk):
        y = torch.empty_like(x)
        lib.addln_set_force_path(path)
        rc = lib.softmax_fwd(P(x), P(y), rows, H, code, S())
        lib.addln_set_force_path(0)
        if rc == mba.binding.ERR_UNSUPPORTED:
            pytest.skip("the forced path cannot run this layout")
        assert rc == 0
        torch.cuda.synchronize()
        ys.append(y)
    no_violation(chk, f"softmax {rows}x{H} {dtype} path {path}")
    assert_close(ys[0], ys[1], f"softmax {rows}x{H} {dtype}")


@pytest.mark.parametrize("dtype", ["fp16", "bf16", "fp32"])
@pytest.mark.parametrize("H", [3, 1000, 1024, 4097])
@pytest.mark.parametrize("aligned", [True, False])
def test_elementwise(chk, dtype, H, aligned):
    rows = 11
    gen = torch.Generator().manual_seed(H)
    x = torch.randn(rows, H, generator=gen).to(TD[dtype]).cuda()
    r = torch.randn(rows, H, generator=gen).to(TD[dtype]).cuda()
    bias = torch.randn(H, generator=gen).cuda()
    if not aligned:
        x, r = misaligned_copy(x), misaligned_copy(r)
    code = mba.binding.DTYPE_CODE[TD[dtype]]
    res = []
    for lib in (mba.lib(), chk):
        y, t, u, a = (torch.empty(rows, H, dtype=TD[dtype], device="cuda") for _ in range(4))
        assert lib.bias_gelu_residual_fwd(P(x), P(r), P(bias), P(y), rows, H, code, S()) == 0
        assert lib.bias_add_fwd(P(x), P(bias), P(t), rows, H, code, S()) == 0
        assert lib.gelu_fwd(P(x), P(u), rows * H, code, S()) == 0
        assert lib.add_fwd(P(x), P(r), P(a), rows * H, code, S()) == 0
        torch.cuda.synchronize()
        res.append((y, t, u, a))
    no_violation(chk, f"elementwise {rows}x{H} {dtype} aligned={aligned}")
    for u, v in zip(*res):
        assert_close(u, v, f"elementwise {rows}x{H} {dtype}")


@pytest.mark.parametrize("dtype", ["fp16", "bf16", "fp32"])
@pytest.mark.parametrize("H", [8, 1000, 1024, 1032, 4096, 8192])
@pytest.mark.parametrize("scalar", [False, True])
@pytest.mark.parametrize("with_dres", [False, True])
def test_backward(chk, dtype, H, scalar, with_dres):
    rows = 45
    gen = torch.Generator().manual_seed(H)
    dy = torch.randn(rows, H, generator=gen).to(TD[dtype]).cuda()
    a = torch.randn(rows, H, generator=gen).to(TD[dtype]).cuda()
    mean = torch.randn(rows, generator=gen).cuda()
    rstd = torch.rand(rows, generator=gen).cuda() + 0.5
    gamma = torch.randn(H, generator=gen).cuda()
    dres = torch.randn(rows, H, generator=gen).to(TD[dtype]).cuda() if with_dres else None
    code = mba.binding.DTYPE_CODE[TD[dtype]]
    res = []
    for lib in (mba.lib(), chk):
        need = lib.add_layernorm_bwd_workspace_size(rows, H, code)
        if need < 0:
            pytest.skip("no backward plan for this shape")
        ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
        dx = torch.empty_like(dy)
        dg = torch.empty(H, device="cuda")
        db = torch.empty(H, device="cuda")
        lib.addln_set_force_path(4 if scalar else 0)
        rc = lib.add_layernorm_bwd(P(dy), P(a), P(mean), P(rstd), P(gamma), P(dres), P(dx), P(dg),
                                   P(db), rows, H, code, P(ws), ws.numel(), S())
        lib.addln_set_force_path(0)
        assert rc == 0, lib.addln_strerror(rc).decode()
        torch.cuda.synchronize()
        res.append((dx, dg, db))
    no_violation(chk, f"backward {rows}x{H} {dtype} scalar={scalar} dres={with_dres}")
    assert_close(res[0][0], res[1][0], f"backward dx {rows}x{H} {dtype}")
    # column sums: partials grouped as each build's grid falls, so within
    # 1e-5 of the sum of magnitudes over the rows
    mag = (dy.double().abs().sum(0) * 4).float()
    for u, v in zip(res[0][1:], res[1][1:]):
        assert ((u - v).abs() <= 1e-5 * mag + 1e-6).all(), f"backward columns {rows}x{H} {dtype}"
