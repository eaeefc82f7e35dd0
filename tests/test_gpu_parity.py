"""GPU parity: the CUDA kernels (called through the C ABI) against the fp64
oracle on the same seeded inputs.

Small cases run every kernel path, every output combination and a ragged
tail of rows; the persistent CTA kernels also run with a capped grid so each
CTA walks many rows through its two-stage copy pipeline.  Full-size
workloads run in the launch configuration the benchmark times and every row
of every output is checked.  Besides the element bounds, the fraction of
16-bit Y equal to the exact value rounded to nearest-even is held to a
minimum, so that a systematic one-unit bias cannot pass.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from _parity import (Rounding, assert_a, assert_correctly_rounded, assert_stats, assert_y,
                     over_row_chunks, ulp, Y_TOL)

pytestmark = pytest.mark.gpu

mba = pytest.importorskip("memory_bound_add_gb300")

PATHS = {
    "auto": 0,
    "warp_vec": 1,
    "cta_tma": 2,
    "cta_vec": 3,
    "scalar": 4,
}
TD = synth.TORCH_DTYPES


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from memory_bound_add_gb300.build import build
    build()
    mba.addln_set_force_path(0)
    mba.addln_set_grid_cap(0)
    yield
    mba.addln_set_force_path(0)
    mba.addln_set_grid_cap(0)


def _dev(d):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def run_fused(d, path=0, want_a=True, want_stats=True, grid_cap=0, inplace=None):
    """One add_layernorm_fwd call on device copies of d's inputs."""
    g = _dev(d)
    x, r = g["x"], g["r"]
    rows = x.shape[0]
    y = torch.empty_like(x)
    a = torch.empty_like(x) if want_a else None
    mean = torch.empty(rows, dtype=torch.float32, device="cuda") if want_stats else None
    rstd = torch.empty(rows, dtype=torch.float32, device="cuda") if want_stats else None
    if inplace == "y=x":
        y = x
    elif inplace == "a=r":
        a = r
    prev = mba.addln_set_force_path(path)
    prev_cap = mba.addln_set_grid_cap(grid_cap)
    try:
        mba.add_layernorm_fwd(x, r, g["gamma"], g["beta"], y, a, mean, rstd, eps=g["eps"])
        name = mba.addln_last_path()
        torch.cuda.synchronize()
    finally:
        mba.addln_set_force_path(prev)
        mba.addln_set_grid_cap(prev_cap)
    assert mba.addln_get_device_error() == 0
    out = {"y": y.cpu(), "a": a.cpu() if a is not None else None,
           "mean": mean.cpu() if mean is not None else None,
           "rstd": rstd.cpu() if rstd is not None else None, "path": name}
    return out


def check(w, d, out, what, rows=None):
    x, r = d["x"], d["r"]
    if rows is not None:
        x, r = x[rows], r[rows]
    ref = oracle.oracle_add_layernorm(x, r, d["gamma"], d["beta"], d["eps"], w.dtype)
    sel = (lambda t: t[rows]) if rows is not None else (lambda t: t)
    assert_y(sel(out["y"]), ref["y"], w.dtype, what)
    assert_correctly_rounded(sel(out["y"]), ref["y"], w.dtype, what)
    if out["a"] is not None:
        assert_a(sel(out["a"]), ref["a"], what)
    if out["mean"] is not None:
        assert_stats(sel(out["mean"]), sel(out["rstd"]), ref["mean"], ref["rstd"], what)
    return ref


def _supported(path, w):
    vec_ok = (w.H * w.elem_bytes) % 16 == 0
    if path == "warp_vec":
        return vec_ok and w.H <= 1024
    if path in ("cta_tma", "cta_vec"):
        return vec_ok
    return True


# ------------------------------------------------------------- small cases
SMALL_ROWS = 301  # not a multiple of the 8 rows a warp-per-row CTA covers


@pytest.mark.parametrize("name", synth.PRIMARY + synth.TAILS)
@pytest.mark.parametrize("path", list(PATHS))
def test_small_all_paths(name, path):
    w = synth.with_rows(synth.get(name), SMALL_ROWS)
    if not _supported(path, w):
        pytest.skip("path cannot run this row layout")
    d = synth.make_inputs(w, seed=1)
    out = run_fused(d, PATHS[path])
    check(w, d, out, f"{name}/{path}/{out['path']}")


@pytest.mark.parametrize("name", ["pages_2048x4096_fp16", "large_32768x8192_bf16",
                                  "tail_4096x1002_fp32", "cancel_65536x1000_bf16"])
@pytest.mark.parametrize("path", ["cta_tma", "cta_vec", "scalar"])
@pytest.mark.parametrize("cap", [1, 7, 19])
def test_persistent_grid_walks_many_rows(name, path, cap):
    w = synth.with_rows(synth.get(name), 150)
    if not _supported(path, w):
        pytest.skip("path cannot run this row layout")
    if path == "scalar" and w.H <= 1024:
        pytest.skip("scalar path is warp-per-row at this H")
    d = synth.make_inputs(w, seed=2)
    out = run_fused(d, PATHS[path], grid_cap=cap)
    check(w, d, out, f"{name}/{path}/cap{cap}")


@pytest.mark.parametrize("want_a,want_stats", [(False, False), (True, False), (False, True)])
@pytest.mark.parametrize("name", ["tiny_64x768_fp32", "pages_2048x4096_fp16",
                                  "tail_4096x999_bf16"])
def test_output_combinations(name, want_a, want_stats):
    w = synth.with_rows(synth.get(name), 77)
    d = synth.make_inputs(w, seed=3)
    out = run_fused(d, 0, want_a=want_a, want_stats=want_stats)
    check(w, d, out, f"{name}/a{int(want_a)}s{int(want_stats)}")


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("H", [1, 2, 7, 8, 9, 31, 32, 33, 255, 257, 1000, 1001, 1023, 1024, 1025,
                               1032, 2048, 2056, 4095, 4097, 4104, 8192, 12288])
@pytest.mark.parametrize("rows", [1, 3, 33])
def test_shape_sweep(dtype, H, rows):
    w = synth.custom(rows, H, dtype, x_dist=(3.0, 2.0), want_resid=True, want_stats=True)
    d = synth.make_inputs(w, seed=H * 7 + rows)
    out = run_fused(d, 0)
    check(w, d, out, f"{rows}x{H} {dtype} {out['path']}")


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
def test_maximum_hidden(dtype):
    H = mba.addln_max_hidden(mba.binding.DTYPE_CODE[TD[dtype]])
    w = synth.custom(5, H, dtype, want_resid=True, want_stats=True)
    d = synth.make_inputs(w, seed=4)
    for path in ("auto", "scalar"):
        out = run_fused(d, PATHS[path])
        check(w, d, out, f"maxH {dtype} {path} {out['path']}")


def test_hidden_above_maximum_is_rejected():
    H = mba.addln_max_hidden(mba.BF16) + 8
    x = torch.zeros(2, H, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(H, device="cuda")
    with pytest.raises(mba.AddLNError) as e:
        mba.add_layernorm(x, x.clone(), g, g.clone())
    assert e.value.code == mba.binding.ERR_SHAPE


# ---------------------------------------------------------------- edge cases
@pytest.mark.parametrize("name", ["tiny_64x768_fp32", "pages_2048x4096_fp16",
                                  "tail_4096x1001_bf16"])
@pytest.mark.parametrize("mode", ["y=x", "a=r"])
def test_in_place(name, mode):
    w = synth.with_rows(synth.get(name), 40)
    d = synth.make_inputs(w, seed=5)
    out = run_fused(d, 0, inplace=mode)
    check(w, d, out, f"{name} in place {mode}")


@pytest.mark.parametrize("dtype,H", [("bf16", 4096), ("fp16", 768), ("fp32", 2048)])
def test_misaligned_pointers_take_element_path(dtype, H):
    rows = 37
    w = synth.custom(rows, H, dtype, want_resid=True, want_stats=True)
    d = synth.make_inputs(w, seed=6)
    n = rows * H
    xb = torch.empty(n + 8, dtype=TD[dtype], device="cuda")
    rb = torch.empty(n + 8, dtype=TD[dtype], device="cuda")
    x = xb[1:1 + n].view(rows, H)
    r = rb[1:1 + n].view(rows, H)
    x.copy_(d["x"].cuda())
    r.copy_(d["r"].cuda())
    y = torch.empty_like(x)
    a = torch.empty_like(x)
    mean = torch.empty(rows, device="cuda")
    rstd = torch.empty(rows, device="cuda")
    g, b = d["gamma"].cuda(), d["beta"].cuda()
    prev = mba.addln_set_force_path(mba.PATH_CTA_TMA)
    try:
        with pytest.raises(mba.AddLNError) as e:
            mba.add_layernorm_fwd(x, r, g, b, y, a, mean, rstd, eps=d["eps"])
        assert e.value.code == mba.binding.ERR_UNSUPPORTED
    finally:
        mba.addln_set_force_path(prev)
    mba.add_layernorm_fwd(x, r, g, b, y, a, mean, rstd, eps=d["eps"])
    assert "scalar" in mba.addln_last_path()
    torch.cuda.synchronize()
    out = {"y": y.cpu(), "a": a.cpu(), "mean": mean.cpu(), "rstd": rstd.cpu()}
    check(w, d, out, f"misaligned {dtype} {H}")


def test_zero_rows_is_a_noop():
    x = torch.empty(0, 768, dtype=torch.float16, device="cuda")
    g = torch.ones(768, device="cuda")
    y, _, _, _ = mba.add_layernorm(x, x, g, g)
    assert y.shape == (0, 768)


@pytest.mark.parametrize("name", ["tiny_64x768_fp32", "pages_2048x4096_fp16",
                                  "tail_4096x999_bf16", "large_32768x8192_bf16"])
def test_outputs_do_not_write_outside_their_rows(name):
    w = synth.with_rows(synth.get(name), 21)
    d = synth.make_inputs(w, seed=7)
    g = _dev(d)
    rows, H = w.rows, w.H
    pad = 128
    sentinel = -12345.0
    ybuf = torch.full((rows * H + 2 * pad,), sentinel, dtype=TD[w.dtype], device="cuda")
    abuf = torch.full((rows * H + 2 * pad,), sentinel, dtype=TD[w.dtype], device="cuda")
    sbuf = torch.full((2 * rows + 4 * pad,), sentinel, dtype=torch.float32, device="cuda")
    y = ybuf[pad:pad + rows * H].view(rows, H)
    a = abuf[pad:pad + rows * H].view(rows, H)
    mean = sbuf[pad:pad + rows]
    rstd = sbuf[3 * pad + rows:3 * pad + 2 * rows]
    mba.add_layernorm_fwd(g["x"], g["r"], g["gamma"], g["beta"], y, a, mean, rstd, eps=g["eps"])
    torch.cuda.synchronize()
    for buf in (ybuf, abuf):
        assert torch.all(buf[:pad] == sentinel) and torch.all(buf[-pad:] == sentinel)
    assert torch.all(sbuf[:pad] == sentinel)
    assert torch.all(sbuf[pad + rows:3 * pad + rows] == sentinel)
    assert torch.all(sbuf[3 * pad + 2 * rows:] == sentinel)
    out = {"y": y.cpu(), "a": a.cpu(), "mean": mean.cpu(), "rstd": rstd.cpu()}
    check(w, d, out, f"{name} canary")


def test_constant_rows_are_exact():
    # a constant row: mean is the constant, the variance 0, and Y is beta
    # rounded to the dtype, on every kernel path
    w = synth.with_rows(synth.get("cancel_65536x1000_bf16"), 400)
    d = synth.make_inputs(w, seed=8)
    cr = d["const_rows"]
    assert len(cr) == 4
    for path in ("auto", "cta_tma", "cta_vec", "scalar"):
        out = run_fused(d, PATHS[path])
        beta_bf16 = d["beta"].to(torch.bfloat16)
        for i in cr:
            assert torch.equal(out["y"][i], beta_bf16), path
            assert out["mean"][i].item() == d["x"][i, 0].float().item(), path
        check(w, d, out, f"constant rows {path}")


def test_deterministic_bitwise():
    w = synth.with_rows(synth.get("large_32768x8192_bf16"), 200)
    d = synth.make_inputs(w, seed=9)
    o1 = run_fused(d, 0)
    o2 = run_fused(d, 0)
    assert torch.equal(o1["y"], o2["y"]) and torch.equal(o1["a"], o2["a"])


# ------------------------------------------------------- unfused baseline
@pytest.mark.parametrize("name", synth.PRIMARY + synth.TAILS)
def test_unfused_chain_matches_oracle_with_rounded_A(name):
    w = synth.with_rows(synth.get(name), 129)
    d = synth.make_inputs(w, seed=10)
    g = _dev(d)
    y, a, mean, rstd = mba.add_then_layernorm(g["x"], g["r"], g["gamma"], g["beta"], eps=g["eps"],
                                              want_stats=True)
    torch.cuda.synchronize()
    ref = oracle.oracle_add_layernorm(d["x"], d["r"], d["gamma"], d["beta"], d["eps"], w.dtype,
                                      round_A=True)
    assert_a(a.cpu(), ref["a"], f"{name} unfused A")
    assert_y(y.cpu(), ref["y"], w.dtype, f"{name} unfused Y")
    assert_stats(mean.cpu(), rstd.cpu(), ref["mean"], ref["rstd"], f"{name} unfused stats")


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("n", [1, 7, 8, 4097, 1 << 20, (1 << 20) + 3])
def test_add_kernel(dtype, n):
    g = torch.Generator().manual_seed(n)
    x = (torch.randn(n, generator=g) * 3).to(TD[dtype])
    r = torch.randn(n, generator=g).to(TD[dtype])
    a = torch.empty_like(x, device="cuda")
    mba.add_fwd(x.cuda(), r.cuda(), a)
    torch.cuda.synchronize()
    assert_a(a.cpu(), oracle.oracle_add(x, r, dtype, round_A=True), f"add {dtype} {n}")


# -------------------------------------------------------- bounded waits
def test_wait_timeout_sets_device_error_and_recovers():
    w = synth.with_rows(synth.get("pages_2048x4096_fp16"), 64)
    d = synth.make_inputs(w, seed=11)
    g = _dev(d)
    y = torch.empty_like(g["x"])
    prev_path = mba.addln_set_force_path(mba.PATH_CTA_TMA)
    prev_limit = mba.addln_set_wait_limit_ns(0)
    try:
        mba.add_layernorm_fwd(g["x"], g["r"], g["gamma"], g["beta"], y, eps=g["eps"])
        assert mba.addln_get_device_error() == mba.binding.ERR_DEVICE_TIMEOUT
    finally:
        mba.addln_set_wait_limit_ns(prev_limit)
        mba.addln_set_force_path(prev_path)
    assert mba.addln_get_device_error() == 0        # read-and-clear
    out = run_fused(d, 0, want_a=False, want_stats=False)
    check(w, d, out, "after timeout")


# ------------------------------------------------------------ full sizes
def check_every_row(w, d, out, what):
    """Every row of a full-size call against the oracle, in row chunks: Y
    within its bound, A bit-exact, mean and rstd within theirs, and the
    correctly rounded fraction of 16-bit Y over the whole output."""
    want_a, want_stats = out["a"] is not None, out["mean"] is not None

    def one(lo, hi):
        ref = oracle.oracle_add_layernorm(d["x"][lo:hi], d["r"][lo:hi], d["gamma"], d["beta"],
                                          d["eps"], w.dtype, want_a=want_a, want_stats=want_stats)
        tag = f"{what} rows [{lo}, {hi})"
        assert_y(out["y"][lo:hi], ref["y"], w.dtype, tag)
        if want_a:
            assert_a(out["a"][lo:hi], ref["a"], tag)
        if want_stats:
            assert_stats(out["mean"][lo:hi], out["rstd"][lo:hi], ref["mean"], ref["rstd"], tag)
        rnd = Rounding(w.dtype)
        rnd.add(out["y"][lo:hi], ref["y"])
        return rnd

    total = Rounding(w.dtype, what)
    for r in over_row_chunks(w.rows, w.H, one):
        for k in ("n", "correct", "above", "below"):
            setattr(total, k, getattr(total, k) + getattr(r, k))
    total.check()
    return total


@pytest.mark.slow
@pytest.mark.parametrize("name", synth.PRIMARY + synth.TAILS)
def test_full_size_every_row(name):
    w = synth.get(name)
    d = synth.make_inputs(w, seed=0)
    out = run_fused(d, 0, want_a=w.want_resid, want_stats=w.want_stats)
    check_every_row(w, d, out, f"{name} full size ({out['path']})")
    for i in d["const_rows"]:
        assert torch.equal(out["y"][i], d["beta"].to(TD[w.dtype]))


@pytest.mark.parametrize("name,rows", [("tiny_64x768_fp32", 64), ("bert_base_4096x768_fp16", 3000),
                                       ("pages_2048x4096_fp16", 64), ("tail_4096x999_bf16", 40)])
@pytest.mark.parametrize("path", ["auto", "cta_vec", "scalar"])
def test_nan_and_inf_stay_in_their_row(name, rows, path):
    # a NaN in one row of X and an infinity in another row of R make those
    # rows' Y NaN (the definition's mean and variance are NaN there) and
    # leave every other row as the oracle computes it; rows 0 and 1 share a
    # warp on the two-rows-a-warp path
    w = synth.with_rows(synth.get(name), rows)
    if not _supported(path, w):
        pytest.skip("path does not take this shape")
    d = synth.make_inputs(w, seed=16 + rows)
    d["x"][0, w.H // 3] = float("nan")
    d["r"][rows - 1, w.H - 1] = float("inf")
    out = run_fused(d, PATHS[path], want_a=True, want_stats=True)
    for i in (0, rows - 1):
        assert torch.isnan(out["y"][i]).all(), (i, out["path"])
        assert torch.isnan(out["mean"][i]) or torch.isinf(out["mean"][i]), (i, out["path"])
    keep = np.arange(1, rows - 1)
    check(w, d, out, f"{name} x{rows} NaN/inf rows {out['path']}", rows=keep)


@pytest.mark.parametrize("H", [768, 4096])
def test_eps_zero_constant_row_is_nan_like_the_definition(H):
    # eps = 0 is accepted: a constant row is 0/0 (NaN Y, rstd = inf, the mean
    # exact), every other row is normalised as usual
    w = synth.custom(6, H, "fp16", eps=0.0, want_resid=True, want_stats=True)
    d = synth.make_inputs(w, seed=14)
    d["x"][2] = 1.5
    d["r"][2] = 0.0
    for path in ("auto", "cta_vec", "scalar"):
        out = run_fused(d, PATHS[path])
        ref = oracle.oracle_add_layernorm(d["x"], d["r"], d["gamma"], d["beta"], 0.0, "fp16")
        assert torch.isnan(out["y"][2]).all() and out["rstd"][2].item() == float("inf")
        assert out["mean"][2].item() == 1.5
        keep = [0, 1, 3, 4, 5]
        assert_y(out["y"][keep], ref["y"][keep], "fp16", f"eps 0 {path}")
        assert_stats(out["mean"][keep], out["rstd"][keep], ref["mean"][keep], ref["rstd"][keep])


# ------------------------------------------- programmatic dependent launch
CHAIN_STEPS = 24


def oracle_chain(d, dtype, steps):
    """The layer chain as defined: layer l normalises X_l + R, and its Y,
    stored in the I/O dtype (rounded to nearest-even), is X_{l+1}.  Returns
    the exact fp64 Y of every layer."""
    x = d["x"]
    ys = []
    for _ in range(steps):
        y = oracle.oracle_add_layernorm(x, d["r"], d["gamma"], d["beta"], d["eps"], dtype,
                                        want_a=False, want_stats=False)["y"]
        ys.append(y)
        x = torch.from_numpy(oracle.oracle_round(y, dtype)).to(TD[dtype])
    return ys


def chain_violations(y_gpu, y_ref, dtype):
    """Layer l of the chain: the stated bound, widened to two units in the
    last place.  The GPU chain's X_l may differ from the oracle chain's in the
    few elements where an earlier layer's output was faithfully but not
    correctly rounded (one unit); normalisation carries such a difference on
    scaled by gamma_j * rstd (about 1), so a layer's output may be one unit
    from its own exact value plus one carried unit."""
    yg = y_gpu.double().numpy()
    err = np.abs(yg - y_ref)
    if dtype == "fp32":
        bound = 2 * Y_TOL["fp32"] * (1 + np.abs(y_ref))
    else:
        bound = np.maximum(Y_TOL[dtype], 2 * ulp(y_ref, dtype))
    return ~(err <= bound)


@pytest.mark.parametrize("name", ["bert_base_4096x768_fp16", "pages_2048x4096_fp16",
                                  "tail_4096x1001_bf16"])
def test_dependent_chain_keeps_order_under_pdl(name):
    # each step reads the previous step's Y as its X: a kernel that touched
    # memory before the previous grid finished would change the result.
    # Every layer of every mode is checked against the oracle's chain.
    w = synth.with_rows(synth.get(name), 256)
    host = synth.make_inputs(w, seed=12)
    d = _dev(host)

    def chain():
        x = d["x"].clone()
        ys = []
        for _ in range(CHAIN_STEPS):
            y = torch.empty_like(x)
            mba.add_layernorm_fwd(x, d["r"], d["gamma"], d["beta"], y, eps=d["eps"])
            ys.append(y)
            x = y
        return ys

    ref = oracle_chain(host, w.dtype, CHAIN_STEPS)
    results = {}
    for pdl in (0, 1):
        prev = mba.addln_set_pdl(pdl)
        try:
            eager = chain()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                graphed = chain()
            g.replay()
            torch.cuda.synchronize()
        finally:
            mba.addln_set_pdl(prev)
        assert mba.addln_get_device_error() == 0
        for mode, ys in (("eager", eager), ("graph", graphed)):
            for l, (yg, yr) in enumerate(zip(ys, ref)):
                bad = chain_violations(yg.cpu(), yr, w.dtype)
                assert not bad.any(), (f"{name} pdl={pdl} {mode} layer {l}: {int(bad.sum())} "
                                       f"outputs out of bound")
        results[pdl] = [y.cpu() for y in eager]
        assert all(torch.equal(a, b) for a, b in zip(eager, graphed)), \
            f"pdl={pdl}: graph differs from eager"
    assert all(torch.equal(a, b) for a, b in zip(results[0], results[1]))
    # the first layer has the oracle's own input: the single-step bounds hold
    assert_y(results[1][0], ref[0], w.dtype, f"{name} chain layer 0")
    assert_correctly_rounded(results[1][0], ref[0], w.dtype, f"{name} chain layer 0")


@pytest.mark.parametrize("warp_rows", [1, 2])
@pytest.mark.parametrize("name,rows", [("bert_base_4096x768_fp16", 777), ("cancel_65536x1000_bf16", 1201),
                                       ("tiny_64x768_fp32", 63), ("bert_base_4096x768_fp16", 1)])
@pytest.mark.parametrize("want_a,want_stats", [(False, False), (True, True)])
def test_rows_per_warp(name, rows, warp_rows, want_a, want_stats):
    # one or two rows a warp on the warp-per-row vector path; an odd row
    # count leaves the last warp a single live row
    w = synth.with_rows(synth.get(name), rows)
    d = synth.make_inputs(w, seed=15 + rows)
    prev = mba.addln_set_warp_rows(warp_rows)
    try:
        out = run_fused(d, 0, want_a=want_a, want_stats=want_stats)
    finally:
        mba.addln_set_warp_rows(prev)
    nv = (w.H // (4 if w.dtype == "fp32" else 8) + 31) // 32
    two = warp_rows == 2 and nv in (3, 4)
    assert out["path"].startswith("warp_vec2" if two else "warp_vec_"), out["path"]
    check(w, d, out, f"{name} x{rows} warp_rows={warp_rows} {out['path']}")


@pytest.mark.parametrize("offset", [-5, -1, 0, 3])
@pytest.mark.parametrize("warp_rows", [1, 2])
def test_warp_cta_size_switch(offset, warp_rows):
    # the warp-per-row kernels take one-warp CTAs while four-warp CTAs
    # would be fewer than the SMs (rows < 4 x SMs x rows-a-warp), four-warp
    # CTAs from there on: both sides of the switch and the rows at it
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rows = 4 * sms * warp_rows + offset
    w = synth.with_rows(synth.get("bert_base_4096x768_fp16"), rows)
    d = synth.make_inputs(w, seed=21 + rows)
    prev = mba.addln_set_warp_rows(warp_rows)
    try:
        out = run_fused(d, 0, want_a=True, want_stats=True)
    finally:
        mba.addln_set_warp_rows(prev)
    check(w, d, out, f"bert x{rows} warp_rows={warp_rows} {out['path']}")


@pytest.mark.parametrize("threads", [128, 256, 512])
@pytest.mark.parametrize("stages", [1, 2, 3, 4])
def test_tma_tuning_shapes(threads, stages):
    w = synth.with_rows(synth.get("pages_2048x4096_fp16"), 150)
    d = synth.make_inputs(w, seed=13)
    prev = mba.addln_set_cta_shape(threads, stages)
    try:
        for cap in (0, 7):
            out = run_fused(d, 0, grid_cap=cap)
            assert out["path"] == f"cta_tma_t{threads}_nv{4096 // 8 // threads}"
            check(w, d, out, f"tma t{threads} s{stages} cap{cap}")
    finally:
        mba.addln_set_cta_shape(0, 0)


def test_shared_memory_sizes_in_any_order():
    # the same kernels at large, small, then large shared-memory footprints
    for H in (32768, 12288, 32768, 8192, 30000):
        w = synth.custom(3, H, "bf16", want_resid=True, want_stats=True)
        d = synth.make_inputs(w, seed=H)
        for path in ("auto", "scalar"):
            out = run_fused(d, PATHS[path])
            check(w, d, out, f"order H={H} {path} {out['path']}")
