"""GPU parity of the fused row softmax (softmax_fwd through the C ABI)
against the fp64 oracle on the same seeded inputs: every kernel path, a shape
sweep across the warp / CTA boundary and the ragged tails, misaligned rows,
in place, extreme values, the bounded-wait timeout, and every row of the
full-size workloads in the benchmark's launch configuration, with the
correctly rounded fraction of 16-bit outputs held to a minimum."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from _parity import CR_MIN_SOFTMAX, Rounding, assert_softmax, over_row_chunks

pytestmark = pytest.mark.gpu
mba = pytest.importorskip("memory_bound_add_gb300")
TD = synth.TORCH_DTYPES


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from memory_bound_add_gb300.build import build
    build()
    mba.addln_set_force_path(0)
    yield
    mba.addln_set_force_path(0)


def run(x_host, path=0, grid_cap=0, inplace=False):
    x = x_host.cuda()
    y = x if inplace else torch.empty_like(x)
    prev = mba.addln_set_force_path(path)
    prev_cap = mba.addln_set_grid_cap(grid_cap)
    try:
        mba.softmax_fwd(x, y)
        name = mba.addln_last_path()
        torch.cuda.synchronize()
    finally:
        mba.addln_set_force_path(prev)
        mba.addln_set_grid_cap(prev_cap)
    assert mba.addln_get_device_error() == 0
    return y.cpu(), name


def check(x_host, dtype, y, what, rows=None):
    xs = x_host if rows is None else x_host[rows]
    ref = oracle.oracle_softmax(xs, dtype)["y"]
    assert_softmax(y if rows is None else y[rows], ref, dtype, what)


PATHS = {"auto": 0, "warp_vec": 1, "cta_tma": 2, "scalar": 4}


def _ok(path, H, dtype):
    vec = (H * (4 if dtype == "fp32" else 2)) % 16 == 0
    if path == "warp_vec":
        return vec and H <= 1024
    if path == "cta_tma":
        return vec
    return True


@pytest.mark.parametrize("name", synth.SOFTMAX_NAMES)
@pytest.mark.parametrize("path", list(PATHS))
def test_small_all_paths(name, path):
    w = synth.with_rows(synth.get(name), 203)
    if not _ok(path, w.H, w.dtype):
        pytest.skip("path cannot run this row layout")
    d = synth.make_inputs(w, seed=1)
    y, p = run(d["x"], PATHS[path])
    check(d["x"], w.dtype, y, f"{name}/{path}/{p}")


@pytest.mark.parametrize("name", synth.SOFTMAX_NAMES)
@pytest.mark.parametrize("path", list(PATHS))
def test_nan_stays_in_its_row(name, path):
    # a NaN in one row makes that row's y NaN (its maximum and sum are NaN)
    # and leaves the neighbouring rows as the oracle computes them
    w = synth.with_rows(synth.get(name), 37)
    if not _ok(path, w.H, w.dtype):
        pytest.skip("path cannot run this row layout")
    d = synth.make_inputs(w, seed=9)
    d["x"][5, w.H // 2] = float("nan")
    y, p = run(d["x"], PATHS[path])
    assert torch.isnan(y[5]).all(), p
    keep = np.array([i for i in range(37) if i != 5])
    check(d["x"], w.dtype, y, f"{name}/{path}/{p} NaN row", rows=keep)


@pytest.mark.parametrize("dtype", ["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("H", [1, 2, 7, 8, 33, 257, 1000, 1024, 1025, 4096, 4097, 12288, 32000])
def test_shape_sweep(dtype, H):
    if H > mba.addln_max_hidden(mba.binding.DTYPE_CODE[TD[dtype]]):
        pytest.skip("above the maximum H for this dtype")
    w = synth.custom(5, H, dtype, x_dist=(1.0, 3.0), op="softmax")
    d = synth.make_inputs(w, seed=H)
    for path in ("auto", "scalar"):
        y, p = run(d["x"], PATHS[path])
        check(d["x"], dtype, y, f"5x{H} {dtype} {p}")


@pytest.mark.parametrize("path", ["cta_tma", "scalar"])
@pytest.mark.parametrize("cap", [1, 7])
def test_persistent_grid_walks_many_rows(path, cap):
    w = synth.with_rows(synth.get("softmax_vocab_4096x32000_bf16"), 40)
    d = synth.make_inputs(w, seed=2)
    y, p = run(d["x"], PATHS[path], grid_cap=cap)
    check(d["x"], w.dtype, y, f"vocab {path} cap{cap} {p}")


@pytest.mark.parametrize("dtype,H", [("fp16", 1024), ("bf16", 4096), ("fp32", 2048)])
def test_in_place_and_misaligned(dtype, H):
    w = synth.custom(33, H, dtype, x_dist=(0.0, 2.0), op="softmax")
    d = synth.make_inputs(w, seed=3)
    y, p = run(d["x"], inplace=True)
    check(d["x"], dtype, y, f"in place {p}")
    n = 33 * H
    buf = torch.empty(n + 8, dtype=TD[dtype], device="cuda")
    x = buf[1:1 + n].view(33, H)
    x.copy_(d["x"].cuda())
    yo = torch.empty_like(x)
    mba.softmax_fwd(x, yo)
    assert "scalar" in mba.addln_last_path()
    torch.cuda.synchronize()
    check(d["x"], dtype, yo.cpu(), "misaligned")


def test_extreme_values():
    x = torch.zeros(4, 2048)
    x[0, :] = 1e4
    x[0, 5] = 1e4 + 1.0                     # large magnitudes: no overflow
    x[1, :] = -float("inf")
    x[1, 100] = 0.0                         # a single finite entry takes all
    x[2, ::2] = -1e4                        # half the row underflows to 0
    x[3, 1024:] = -float("inf")             # whole slices of -inf
    for path in ("auto", "scalar"):
        y, p = run(x, PATHS[path])
        check(x, "fp32", y, f"extreme {p}")
        assert torch.isfinite(y).all()


def test_constant_row_is_uniform():
    x = torch.full((3, 4096), 2.5, dtype=torch.bfloat16)
    y, p = run(x)
    check(x, "bf16", y, f"constant rows {p}")
    assert torch.allclose(y.double().sum(dim=1), torch.ones(3, dtype=torch.float64), atol=1e-2)


def test_wait_timeout_sets_device_error_and_recovers():
    w = synth.with_rows(synth.get("softmax_vocab_4096x32000_bf16"), 16)
    d = synth.make_inputs(w, seed=4)
    x = d["x"].cuda()
    y = torch.empty_like(x)
    prev_path = mba.addln_set_force_path(mba.PATH_CTA_TMA)
    prev_limit = mba.addln_set_wait_limit_ns(0)
    try:
        mba.softmax_fwd(x, y)
        assert mba.addln_get_device_error() == mba.binding.ERR_DEVICE_TIMEOUT
    finally:
        mba.addln_set_wait_limit_ns(prev_limit)
        mba.addln_set_force_path(prev_path)
    assert mba.addln_get_device_error() == 0
    y2, _ = run(d["x"])
    check(d["x"], w.dtype, y2, "after timeout")


@pytest.mark.slow
@pytest.mark.parametrize("name", synth.SOFTMAX_NAMES)
def test_full_size_every_row(name):
    w = synth.get(name)
    d = synth.make_inputs(w, seed=0)
    y, p = run(d["x"])
    what = f"{name} full size ({p})"

    def one(lo, hi):
        ref = oracle.oracle_softmax(d["x"][lo:hi], w.dtype)["y"]
        assert_softmax(y[lo:hi], ref, w.dtype, f"{what} rows [{lo}, {hi})")
        rnd = Rounding(w.dtype)
        rnd.add(y[lo:hi], ref)
        return rnd

    total = Rounding(w.dtype, what)
    for r in over_row_chunks(w.rows, w.H, one):
        for k in ("n", "correct", "above", "below"):
            setattr(total, k, getattr(total, k) + getattr(r, k))
    total.check(CR_MIN_SOFTMAX)
    assert torch.isfinite(y).all()


def test_shared_memory_sizes_in_any_order():
    # large, small, then large again on the same kernels: the dynamic shared
    # memory limit of a kernel must never be left below a later launch's need
    for H in (32000, 12288, 32000, 2048, 30000):
        w = synth.custom(3, H, "bf16", x_dist=(0.0, 2.0), op="softmax")
        d = synth.make_inputs(w, seed=H)
        for path in ("cta_tma", "scalar"):
            y, p = run(d["x"], PATHS[path])
            check(d["x"], "bf16", y, f"order H={H} {p}")


@pytest.mark.parametrize("threads", [0, 512])
def test_long_rows_both_variants(threads):
    # 0: the staged row is re-read from shared memory (two passes);
    # 512: the row is held in registers by 512 threads x 8 vectors
    w = synth.with_rows(synth.get("softmax_vocab_4096x32000_bf16"), 23)
    d = synth.make_inputs(w, seed=5)
    prev = mba.addln_set_cta_shape(threads, 0)
    try:
        y, p = run(d["x"])
    finally:
        mba.addln_set_cta_shape(0, 0)
    assert p == ("softmax_cta_tma_t512_nv8" if threads == 512 else "softmax_cta_tma_smem_t256")
    check(d["x"], w.dtype, y, p)
